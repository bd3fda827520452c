"""Host-side argument checks of every entry point after gdn_forward (no GPU needed).

Each call below gets fake, never-dereferenced device addresses and one bad argument,
and must return the status include/gdn.h documents for it before any CUDA call.  The
empty cases (no tokens, no sequences, no blocks) return GDN_OK on the host, also before
any CUDA call.  The tests skip where a CUDA device is visible: there a call that passed
its checks by mistake would launch on the fake addresses.
"""
import ctypes

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device addresses: host-only machines")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 0, -1, -2, -3, -6


@pytest.fixture(scope="module")
def gdn():
    import __graft_entry__
    __graft_entry__._builder().build()
    import gated_deltanet_backward_gb300 as g
    return g


class Fake:
    """Distinct 256-byte-aligned addresses, 1 GiB apart, so that no two overlap."""

    def __init__(self):
        self.n = 0

    def __call__(self):
        self.n += 1
        return (1 << 40) + self.n * (1 << 30)


def _call(fn, order, args, **over):
    a = dict(args)
    for k, v in over.items():
        assert k in a, k
        a[k] = v
    return fn(*[a[k] for k in order])


# --- gdn_backward --------------------------------------------------------------------

BWD_ORDER = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
             "beta_ld", "a_log", "dt", "cu", "coff", "S0", "dO", "dO_ld", "dS_T", "saved",
             "dq", "dq_ld", "dk", "dk_ld", "dv", "dv_ld", "dalpha", "dalpha_ld", "dbeta",
             "dbeta_ld", "da_log", "ddt", "dS0", "ws", "ws_bytes", "flags", "stream"]


def test_backward_checks(gdn):
    f = Fake()
    s = gdn.make_shape(2, 6, 64, 64, 1, 2, 100, "f32")
    ws = gdn.gdn_workspace_bytes(s, True)
    wq, wv = 2 * 64, 6 * 64
    a = dict(shape=ctypes.byref(s), q=f(), q_ld=wq, k=f(), k_ld=wq, v=f(), v_ld=wv, alpha=f(),
             alpha_ld=6, beta=f(), beta_ld=6, a_log=f(), dt=f(), cu=f(), coff=f(), S0=None,
             dO=f(), dO_ld=wv, dS_T=None, saved=f(), dq=f(), dq_ld=wq, dk=f(), dk_ld=wq, dv=f(),
             dv_ld=wv, dalpha=f(), dalpha_ld=6, dbeta=f(), dbeta_ld=6, da_log=f(), ddt=f(),
             dS0=None, ws=f(), ws_bytes=ws, flags=0, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_backward, BWD_ORDER, a, **o)
    assert run(flags=gdn.GDN_FLAG_KEEP_FOR_BACKWARD) == INVALID      # a forward-only flag
    assert run(flags=8) == INVALID                                    # no such flag
    # bf16 saved states: bf16 inputs with Dk, Dv >= 64 only
    assert run(flags=gdn.GDN_FLAG_BF16_SAVED_STATES) == UNSUPPORTED   # fp32 inputs
    s16 = gdn.make_shape(2, 6, 64, 32, 1, 2, 100, "bf16")
    assert run(shape=ctypes.byref(s16), flags=gdn.GDN_FLAG_BF16_SAVED_STATES,
               ws_bytes=gdn.gdn_workspace_bytes(s16, True), dO_ld=6 * 32,
               dv_ld=6 * 32, v_ld=6 * 32) == UNSUPPORTED
    assert run(saved=None) == INVALID                                 # chunks need states
    assert run(ws_bytes=gdn.gdn_workspace_bytes(s, False)) == WORKSPACE
    assert run(dO_ld=wv - 8) == INVALID
    assert run(dq=a["dq"] + 8) == MISALIGNED
    assert run(dalpha_ld=5) == INVALID
    assert run(da_log=None) == INVALID
    assert run(dS0=a["ws"] + 4) == MISALIGNED


# --- gdn_decode_step -----------------------------------------------------------------

DEC_ORDER = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
             "beta_ld", "a_log", "dt", "S_in", "S_out", "o", "o_ld", "stream"]


def test_decode_step_checks(gdn):
    f = Fake()
    s = gdn.make_shape(2, 4, 64, 64, 3, 0, 0, "bf16")   # token and chunk counts are implied
    a = dict(shape=ctypes.byref(s), q=f(), q_ld=128, k=f(), k_ld=128, v=f(), v_ld=256,
             alpha=f(), alpha_ld=4, beta=f(), beta_ld=4, a_log=f(), dt=f(), S_in=None,
             S_out=f(), o=f(), o_ld=256, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_decode_step, DEC_ORDER, a, **o)
    assert run(shape=None) == INVALID
    assert run(S_out=None) == INVALID
    assert run(q_ld=64) == INVALID
    assert run(v_ld=260) == MISALIGNED                  # 520 bytes: not a multiple of 16
    assert run(o=a["o"] + 2) == MISALIGNED
    assert run(beta_ld=3) == INVALID
    bad = gdn.make_shape(2, 4, 48, 64, 3, 0, 0, "bf16")
    assert run(shape=ctypes.byref(bad)) == UNSUPPORTED
    odd = gdn.make_shape(3, 4, 64, 64, 3, 0, 0, "bf16")
    assert run(shape=ctypes.byref(odd)) == INVALID      # Hv not a multiple of Hk
    none = gdn.make_shape(2, 4, 64, 64, 0, 0, 0, "bf16")
    assert run(shape=ctypes.byref(none), S_out=None) == OK


# --- conv1d + SiLU ---------------------------------------------------------------------

CONV_F = ["dtype", "T", "C", "K", "cu", "n", "x", "x_ld", "w", "y", "y_ld", "stream"]
CONV_B = ["dtype", "T", "C", "K", "cu", "n", "x", "x_ld", "w", "dy", "dy_ld", "dx", "dx_ld",
          "dw", "ws", "ws_bytes", "stream"]


def test_conv_checks(gdn):
    f = Fake()
    C, T, K = 64, 100, 4
    a = dict(dtype=1, T=T, C=C, K=K, cu=f(), n=2, x=f(), x_ld=C, w=f(), y=f(), y_ld=C,
             stream=None)
    run = lambda **o: _call(gdn._lib.gdn_conv1d_silu_forward, CONV_F, a, **o)
    assert run(dtype=7) == UNSUPPORTED
    assert run(C=60) == UNSUPPORTED                     # channels in whole 16-byte pieces
    assert run(K=5) == UNSUPPORTED and run(K=0) == UNSUPPORTED
    assert run(n=0) == INVALID                          # tokens without sequences
    assert run(T=-1) == INVALID
    assert run(cu=None) == INVALID
    assert run(cu=a["cu"] + 2) == MISALIGNED
    assert run(w=None) == INVALID
    assert run(x=a["x"] + 8) == MISALIGNED
    assert run(y_ld=C - 8) == INVALID
    assert run(y=a["x"]) == INVALID                     # in place is refused
    assert run(y=a["x"] + 2 * C * 50) == INVALID        # so is any overlap
    assert run(T=0, n=0, cu=None) == OK
    need = gdn.gdn_conv1d_silu_workspace_bytes(T, C, K)
    assert need > 0 and gdn.gdn_conv1d_silu_workspace_bytes(0, C, K) == 0
    b = dict(a, dy=f(), dy_ld=C, dx=f(), dx_ld=C, dw=f(), ws=f(), ws_bytes=need)
    del b["y"], b["y_ld"]
    runb = lambda **o: _call(gdn._lib.gdn_conv1d_silu_backward, CONV_B, b, **o)
    assert runb(ws_bytes=need - 1) == WORKSPACE
    assert runb(ws=None) == WORKSPACE
    assert runb(dx=b["dy"]) == INVALID
    assert runb(dx=b["x"]) == INVALID
    assert runb(dw=b["dw"] + 4) == MISALIGNED
    assert runb(dx_ld=C - 8) == INVALID


# --- gated RMSNorm ---------------------------------------------------------------------

NORM_F = ["dtype", "T", "H", "D", "eps", "o", "o_ld", "z", "z_ld", "gamma", "y", "y_ld",
          "stream"]
NORM_B = ["dtype", "T", "H", "D", "eps", "o", "o_ld", "z", "z_ld", "gamma", "dy", "dy_ld",
          "d_o", "do_ld", "dz", "dz_ld", "dgamma", "ws", "ws_bytes", "stream"]


def test_norm_checks(gdn):
    f = Fake()
    H, D, T = 4, 128, 50
    W = H * D
    a = dict(dtype=0, T=T, H=H, D=D, eps=1e-6, o=f(), o_ld=W, z=f(), z_ld=W, gamma=f(), y=f(),
             y_ld=W, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_gated_rmsnorm_forward, NORM_F, a, **o)
    assert run(eps=-1e-6) == INVALID
    assert run(eps=float("nan")) == INVALID
    assert run(eps=float("inf")) == INVALID
    assert run(D=96) == UNSUPPORTED
    assert run(T=(1 << 31) // W + 1) == UNSUPPORTED     # 32-bit element indices
    assert run(H=0) == INVALID
    assert run(gamma=None) == INVALID
    assert run(y=a["o"]) == INVALID and run(y=a["z"]) == INVALID
    assert run(z_ld=W + 1) == MISALIGNED
    assert run(T=0) == OK
    need = gdn.gdn_gated_rmsnorm_workspace_bytes(D)
    assert need > 0 and gdn.gdn_gated_rmsnorm_workspace_bytes(0) == 0
    b = dict(a, dy=f(), dy_ld=W, d_o=f(), do_ld=W, dz=f(), dz_ld=W, dgamma=f(), ws=f(),
             ws_bytes=need)
    del b["y"], b["y_ld"]
    runb = lambda **o: _call(gdn._lib.gdn_gated_rmsnorm_backward, NORM_B, b, **o)
    assert runb(d_o=b["dz"]) == INVALID
    assert runb(d_o=b["dy"]) == INVALID and runb(dz=b["o"]) == INVALID
    assert runb(ws_bytes=need - 16) == WORKSPACE
    assert runb(dgamma=b["dgamma"] + 4) == MISALIGNED


# --- state composition -----------------------------------------------------------------

COMPOSE = ["n", "Dk", "Dv", "Phi", "S", "R", "out", "transpose", "stream"]


def test_state_compose_checks(gdn):
    f = Fake()
    a = dict(n=8, Dk=128, Dv=128, Phi=f(), S=f(), R=f(), out=f(), transpose=0, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_state_compose, COMPOSE, a, **o)
    assert run(n=-1) == INVALID
    assert run(transpose=2) == INVALID
    assert run(Dk=0) == INVALID and run(Dv=5000) == INVALID
    assert run(n=65536) == UNSUPPORTED
    assert run(Phi=None) == INVALID
    assert run(S=a["S"] + 4) == MISALIGNED
    assert run(out=a["S"]) == INVALID and run(out=a["Phi"]) == INVALID
    assert run(R=a["out"] + 16) == INVALID              # partly overlapping R
    assert run(n=0, Phi=None, S=None, out=None) == OK


# --- KDA -----------------------------------------------------------------------------

KDA_F = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
         "beta_ld", "a_log", "b_alpha", "cu", "S_in", "S_out", "o", "o_ld", "stream"]
KDA_B = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
         "beta_ld", "a_log", "b_alpha", "cu", "S0", "dO", "dO_ld", "dS_T", "dq", "dq_ld", "dk",
         "dk_ld", "dv", "dv_ld", "dalpha", "dalpha_ld", "dbeta", "dbeta_ld", "da_log",
         "db_alpha", "dS0", "ws", "ws_bytes", "stream"]


def test_kda_checks(gdn):
    f = Fake()
    Hk, Hv, Dk, Dv, T = 2, 4, 64, 64, 40
    s = gdn.make_shape(Hk, Hv, Dk, Dv, 2, 0, T, "bf16")   # the chunk count is not used
    wq, wv, wa = Hk * Dk, Hv * Dv, Hv * Dk
    a = dict(shape=ctypes.byref(s), q=f(), q_ld=wq, k=f(), k_ld=wq, v=f(), v_ld=wv, alpha=f(),
             alpha_ld=wa, beta=f(), beta_ld=Hv, a_log=f(), b_alpha=f(), cu=f(), S_in=None,
             S_out=f(), o=f(), o_ld=wv, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_kda_forward, KDA_F, a, **o)
    assert run(alpha_ld=Hv) == INVALID                  # one gate per key channel: Hv*Dk
    assert run(b_alpha=None) == INVALID
    assert run(cu=None) == INVALID
    assert run(cu=a["cu"] + 2) == MISALIGNED
    assert run(S_out=None) == INVALID
    bad = gdn.make_shape(Hk, Hv, 48, Dv, 2, 0, T, "bf16")
    assert run(shape=ctypes.byref(bad)) == UNSUPPORTED
    empty = gdn.make_shape(Hk, Hv, Dk, Dv, 0, 0, 0, "bf16")
    assert run(shape=ctypes.byref(empty), cu=None, S_out=None) == OK
    need = gdn.gdn_kda_backward_workspace_bytes(s)
    assert need > 0 and gdn._lib.gdn_kda_backward_workspace_bytes(None) == 0
    b = dict(a, S0=None, dO=f(), dO_ld=wv, dS_T=None, dq=f(), dq_ld=wq, dk=f(), dk_ld=wq,
             dv=f(), dv_ld=wv, dalpha=f(), dalpha_ld=wa, dbeta=f(), dbeta_ld=Hv, da_log=f(),
             db_alpha=f(), dS0=None, ws=f(), ws_bytes=need)
    for k in ("S_in", "S_out", "o", "o_ld"):
        del b[k]
    runb = lambda **o: _call(gdn._lib.gdn_kda_backward, KDA_B, b, **o)
    assert runb(dalpha_ld=Hv) == INVALID
    assert runb(db_alpha=None) == INVALID and runb(da_log=None) == INVALID
    assert runb(ws_bytes=need - 1) == WORKSPACE
    assert runb(ws=None) == WORKSPACE
    narrow = gdn.make_shape(Hk, Hv, Dk, 16, 2, 0, T, "bf16")
    assert runb(shape=ctypes.byref(narrow)) == UNSUPPORTED    # 32-column state slices
    many = gdn.make_shape(Hk, Hv, Dk, Dv, 65536, 0, 65536, "bf16")
    assert runb(shape=ctypes.byref(many)) == UNSUPPORTED


# --- gdn_forward_gated_rmsnorm -----------------------------------------------------------

FWDN_ORDER = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
              "beta_ld", "a_log", "dt", "cu", "coff", "S0", "o", "o_ld", "S_T", "saved", "z",
              "z_ld", "gamma", "eps", "y", "y_ld", "ws", "ws_bytes", "flags", "stream"]


def test_forward_gated_rmsnorm_checks(gdn):
    f = Fake()
    s = gdn.make_shape(2, 6, 64, 64, 1, 2, 100, "bf16")
    ws = gdn.gdn_workspace_bytes(s, False)
    wq, wv = 2 * 64, 6 * 64
    a = dict(shape=ctypes.byref(s), q=f(), q_ld=wq, k=f(), k_ld=wq, v=f(), v_ld=wv, alpha=f(),
             alpha_ld=6, beta=f(), beta_ld=6, a_log=f(), dt=f(), cu=f(), coff=f(), S0=None,
             o=f(), o_ld=wv, S_T=None, saved=None, z=f(), z_ld=wv, gamma=f(), eps=1e-6, y=f(),
             y_ld=wv, ws=f(), ws_bytes=ws, flags=0, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_forward_gated_rmsnorm, FWDN_ORDER, a, **o)
    assert run(y=None) == INVALID
    assert run(gamma=None) == INVALID
    assert run(z=None) == INVALID
    assert run(eps=-1.0) == INVALID and run(eps=float("nan")) == INVALID
    assert run(y=a["o"]) == INVALID and run(y=a["z"]) == INVALID and run(z=a["o"]) == INVALID
    assert run(z_ld=wv + 1) == MISALIGNED and run(y=a["y"] + 2) == MISALIGNED
    assert run(y_ld=wv - 8) == INVALID
    # the recurrence's own checks come first, as in gdn_forward
    assert run(q=None) == INVALID
    assert run(ws_bytes=ws - 1) == WORKSPACE


# --- gdn_kda_forward_chunked -----------------------------------------------------------

KDAC_ORDER = ["shape", "q", "q_ld", "k", "k_ld", "v", "v_ld", "alpha", "alpha_ld", "beta",
              "beta_ld", "a_log", "b_alpha", "cu", "coff", "S_in", "S_out", "o", "o_ld", "ws",
              "ws_bytes", "stream"]


def test_kda_forward_chunked_checks(gdn):
    f = Fake()
    s = gdn.make_shape(2, 6, 128, 128, 1, 2, 100, "bf16")
    ws = gdn.gdn_kda_forward_chunked_workspace_bytes(s)
    assert ws > 0
    wq, wv = 2 * 128, 6 * 128
    a = dict(shape=ctypes.byref(s), q=f(), q_ld=wq, k=f(), k_ld=wq, v=f(), v_ld=wv, alpha=f(),
             alpha_ld=6 * 128, beta=f(), beta_ld=6, a_log=f(), b_alpha=f(), cu=f(), coff=f(),
             S_in=None, S_out=f(), o=f(), o_ld=wv, ws=f(), ws_bytes=ws, stream=None)
    run = lambda **o: _call(gdn._lib.gdn_kda_forward_chunked, KDAC_ORDER, a, **o)
    assert run(alpha_ld=6 * 128 - 1) == INVALID          # one gate column per key channel
    assert run(b_alpha=None) == INVALID and run(a_log=None) == INVALID
    assert run(coff=None) == INVALID and run(cu=None) == INVALID
    assert run(coff=a["coff"] + 2) == MISALIGNED
    assert run(S_out=None) == INVALID
    assert run(ws_bytes=ws - 1) == WORKSPACE and run(ws=a["ws"] + 16) == WORKSPACE
    assert run(q_ld=wq + 1) == MISALIGNED
    for dt, Dk, Dv in (("f32", 128, 128), ("bf16", 32, 128), ("bf16", 128, 16)):
        s2 = gdn.make_shape(2, 6, Dk, Dv, 1, 2, 100, dt)
        assert gdn.gdn_kda_forward_chunked_workspace_bytes(s2) == 0
        assert run(shape=ctypes.byref(s2)) == UNSUPPORTED
    s3 = gdn.make_shape(2, 6, 128, 128, 0, 0, 0, "bf16")
    assert run(shape=ctypes.byref(s3), cu=None, coff=None, S_out=None) == OK
