"""The Python binding's tensor checks (no GPU needed).

The C ABI sees only pointers and row strides, so the binding checks each tensor before
handing it over: dtype, at least the rows and columns (elements, bytes) the call reads
or writes, and, after every size, that the tensor is on the current CUDA device.  Here
every entry point gets host tensors laid out as a real call lays them out (q, k, v as
column views of one packed projection, states [N, Hv, Dk, Dv], ...).  Such a call passes
every size and dtype check and stops at the device check, which shows that the checks
accept real layouts.  Each test then breaks one property at a time and expects the
check that names it.
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host tensors stand in for device tensors")

ON_DEVICE = "not on the current CUDA device"


@pytest.fixture(scope="module")
def gdn():
    import __graft_entry__
    __graft_entry__._builder().build()
    import gated_deltanet_backward_gb300 as g
    return g


def _fails(fn, *args, match, code=-1, **kw):
    import gated_deltanet_backward_gb300 as g
    with pytest.raises(g.GdnError, match=match) as e:
        fn(*args, **kw)
    assert e.value.code == code, str(e.value)


def _recurrence(gdn, dtype="bf16", Hk=2, Hv=6, D=64, lens=(70, 0, 30)):
    import numpy as np
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, N = int(cu[-1]), len(lens)
    layer = gdn.Layer.create(Hk, Hv, D, D, cu, dtype, device="cpu")
    qkv = torch.zeros(T, 2 * Hk * D + Hv * D, dtype=td)
    a = dict(q=qkv[:, :Hk * D], k=qkv[:, Hk * D:2 * Hk * D], v=qkv[:, 2 * Hk * D:],
             alpha=torch.zeros(T, Hv), beta_raw=torch.zeros(T, Hv), a_log=torch.zeros(Hv),
             dt_bias=torch.zeros(Hv), S0=torch.zeros(N, Hv, D, D),
             o=torch.zeros(T, Hv * D, dtype=td), S_T=torch.zeros(N, Hv, D, D))
    dqkv = torch.zeros_like(qkv)
    g = dict(dO=torch.zeros(T, Hv * D, dtype=td), dS_T=torch.zeros(N, Hv, D, D),
             dq=dqkv[:, :Hk * D], dk=dqkv[:, Hk * D:2 * Hk * D], dv=dqkv[:, 2 * Hk * D:],
             dalpha=torch.zeros(T, Hv), dbeta_raw=torch.zeros(T, Hv), da_log=torch.zeros(Hv),
             ddt_bias=torch.zeros(Hv), dS0=torch.zeros(N, Hv, D, D))
    return layer, a, g, td


def _fwd(gdn, layer, a, **over):
    b = dict(a, **over)
    gdn.gdn_forward(layer.shape, b["q"], b["k"], b["v"], b["alpha"], b["beta_raw"], b["a_log"],
                    b["dt_bias"], b.get("cu", layer.cu_seqlens),
                    b.get("coff", layer.chunk_offsets), b["S0"], b["o"], b["S_T"],
                    b.get("saved", layer.saved_states), layer.ws_fwd, stream=0)


def _bwd(gdn, layer, a, g, **over):
    b = dict(a, **g)
    b.update(over)
    gdn.gdn_backward(layer.shape, b["q"], b["k"], b["v"], b["alpha"], b["beta_raw"],
                     b["a_log"], b["dt_bias"], layer.cu_seqlens, layer.chunk_offsets, b["S0"],
                     b["dO"], b["dS_T"], b.get("saved", layer.saved_states), b["dq"], b["dk"],
                     b["dv"], b["dalpha"], b["dbeta_raw"], b["da_log"], b["ddt_bias"],
                     b["dS0"], layer.ws_bwd, stream=0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forward_and_backward(gdn, dtype):
    layer, a, g, td = _recurrence(gdn, dtype)
    T = a["o"].shape[0]
    _fails(_fwd, gdn, layer, a, match=ON_DEVICE)
    _fails(_bwd, gdn, layer, a, g, match=ON_DEVICE)
    # Layer's own methods marshal the same way
    _fails(layer.forward, a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"], a["a_log"],
           a["dt_bias"], None, a["o"], None, stream=0, train=True, match=ON_DEVICE)
    other = torch.float32 if td == torch.bfloat16 else torch.bfloat16
    _fails(_fwd, gdn, layer, a, q=a["q"].to(other), match="q is torch")
    _fails(_fwd, gdn, layer, a, o=a["o"][:T - 1], match="o is .* needs at least")
    _fails(_fwd, gdn, layer, a, v=a["v"][:, :-1], match="v is .* needs at least")
    _fails(_fwd, gdn, layer, a, alpha=a["alpha"][:, :-1], match="alpha is")
    _fails(_fwd, gdn, layer, a, beta_raw=a["beta_raw"].double(), match="beta_raw is torch")
    _fails(_fwd, gdn, layer, a, a_log=a["a_log"][:-1], match="a_log has")
    _fails(_fwd, gdn, layer, a, S0=a["S0"][:, :-1], match="S0 has")
    _fails(_fwd, gdn, layer, a, S_T=a["S_T"].transpose(2, 3), match="S_T must be contiguous")
    _fails(_fwd, gdn, layer, a, cu=layer.cu_seqlens.long(), match="cu_seqlens is torch")
    _fails(_fwd, gdn, layer, a, coff=layer.chunk_offsets[:-1], match="chunk_offsets has")
    _fails(_fwd, gdn, layer, a, saved=layer.saved_states[:-1], match="saved_states has")
    _fails(_fwd, gdn, layer, a, k=torch.zeros(a["k"].shape[1], T, dtype=td).t(),
           match="k needs contiguous columns")
    _fails(_fwd, gdn, layer, a, q=a["q"].reshape(-1), match="q must be 2-D")
    _fails(_bwd, gdn, layer, a, g, dq=g["dq"][:, 1:], match="dq is")
    _fails(_bwd, gdn, layer, a, g, dalpha=g["dalpha"][:-1], match="dalpha is")
    _fails(_bwd, gdn, layer, a, g, ddt_bias=g["ddt_bias"].half(), match="ddt_bias is torch")
    _fails(_bwd, gdn, layer, a, g, dS0=g["dS0"][:1, :1], match="dS0 has")
    bad = gdn.make_shape(2, 6, 64, 64, 3, 2, 100, 7)
    _fails(gdn.gdn_forward, bad, *([None] * 14), stream=0, match="neither f32 nor bf16",
           code=-2)


def test_noalloc_and_decode(gdn):
    layer, a, _, td = _recurrence(gdn, "bf16")
    s = layer.shape
    _fails(gdn.gdn_forward_noalloc, s, a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"],
           a["a_log"], a["dt_bias"], layer.cu_seqlens, layer.chunk_offsets, a["S0"], a["o"],
           a["S_T"], layer.saved_states, stream=0, match=ON_DEVICE)
    # with no tensors at all the library's own checks answer (the 27B layer's forward
    # needs more scratch than the built-in array holds)
    big = gdn.make_shape(16, 48, 128, 128, 1, 64, 4096, "bf16")
    _fails(gdn.gdn_forward_noalloc, big, *([None] * 13), stream=0, match="GDN_ERR_WORKSPACE",
           code=-6)
    N, Hk, Hv, D = 3, 1, 2, 32
    d = gdn.make_shape(Hk, Hv, D, D, N, N, N, "f32")
    z = lambda *sh: torch.zeros(*sh)
    q, v, o, gt, hv, S = z(N, D), z(N, Hv * D), z(N, Hv * D), z(N, Hv), z(Hv), z(N, Hv, D, D)
    _fails(gdn.gdn_decode_step, d, q, q, v, gt, gt, hv, hv, S, S, o, stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_decode_step, d, q, q, v, gt, gt, hv, hv, None, S, o[:N - 1], stream=0,
           match="o is")
    _fails(gdn.gdn_decode_step, d, q, q, v, gt, gt, hv, hv, None, S[:N - 1], o, stream=0,
           match="S_out has")


def test_conv(gdn):
    T, C, K = 40, 64, 4
    cu = torch.tensor([0, 25, T], dtype=torch.int32)
    x, y = torch.zeros(T, C, dtype=torch.bfloat16), torch.zeros(T, C, dtype=torch.bfloat16)
    w = torch.zeros(C, K)
    ws = torch.zeros(gdn.gdn_conv1d_silu_workspace_bytes(T, C, K), dtype=torch.uint8)
    _fails(gdn.gdn_conv1d_silu_forward, x, w, cu, y, stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_conv1d_silu_backward, x, w, cu, x.clone(), y, torch.zeros(C, K), ws,
           stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_conv1d_silu_forward, x, w, cu, y.float(), stream=0, match="y is torch")
    _fails(gdn.gdn_conv1d_silu_forward, x, w, cu, y[:, :C - 8], stream=0, match="y is")
    _fails(gdn.gdn_conv1d_silu_forward, x.half(), w, cu, y.half(), stream=0,
           match="float32 or bfloat16", code=-2)
    _fails(gdn.gdn_conv1d_silu_forward, x, w.reshape(-1), cu, y, stream=0, match="w must be")
    _fails(gdn.gdn_conv1d_silu_forward, x, w.double(), cu, y, stream=0, match="w is torch")
    _fails(gdn.gdn_conv1d_silu_forward, x, w.t().contiguous().t(), cu, y, stream=0,
           match="w must be contiguous")
    _fails(gdn.gdn_conv1d_silu_backward, x, w, cu, x.clone(), y, torch.zeros(C, K - 1), ws,
           stream=0, match="dw has")
    _fails(gdn.gdn_conv1d_silu_backward, x, w, cu, x[:T - 1], y, None, None, stream=0,
           match="dy is")


def test_norm(gdn):
    T, H, D = 12, 4, 32
    o = torch.zeros(T, H * D, dtype=torch.bfloat16)
    gamma = torch.ones(D)
    ws = torch.zeros(gdn.gdn_gated_rmsnorm_workspace_bytes(D), dtype=torch.uint8)
    _fails(gdn.gdn_gated_rmsnorm_forward, o, o.clone(), gamma, o.clone(), 1e-6, stream=0,
           match=ON_DEVICE)
    _fails(gdn.gdn_gated_rmsnorm_backward, o, o.clone(), gamma, o.clone(), o.clone(),
           o.clone(), 1e-6, torch.zeros(D), ws, stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_gated_rmsnorm_forward, o, o[:, :-8], gamma, o.clone(), 1e-6, stream=0,
           match="z is")
    _fails(gdn.gdn_gated_rmsnorm_forward, o, o.clone(), gamma.bfloat16(), o.clone(), 1e-6,
           stream=0, match="gamma is torch")
    _fails(gdn.gdn_gated_rmsnorm_forward, o, o.clone(), torch.ones(0), o.clone(), 1e-6,
           stream=0, match="gamma must hold")
    _fails(gdn.gdn_gated_rmsnorm_backward, o, o.clone(), gamma, o.clone(), o.clone(),
           o.clone().float(), 1e-6, stream=0, match="dz is torch")
    _fails(gdn.gdn_gated_rmsnorm_backward, o, o.clone(), gamma, o.clone(), o.clone(),
           o.clone(), 1e-6, torch.zeros(D - 1), ws, stream=0, match="dgamma has")


def test_compose(gdn):
    Hv, Dk, Dv = 4, 16, 32
    Phi, S = torch.zeros(1, Hv, Dk, Dk), torch.zeros(1, Hv, Dk, Dv)
    R, out = torch.zeros_like(S), torch.zeros_like(S)
    _fails(gdn.gdn_state_compose, Phi, S, R, out, stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_state_compose, Phi, S, None, out, True, stream=0, match=ON_DEVICE)
    _fails(gdn.gdn_state_compose, Phi[:, :Hv - 1], S, R, out, stream=0, match="Phi has")
    _fails(gdn.gdn_state_compose, Phi.transpose(2, 3), S, R, out, stream=0,
           match="Phi must be contiguous")
    _fails(gdn.gdn_state_compose, Phi, S, R, out[:, :Hv - 1], stream=0, match="out has")
    _fails(gdn.gdn_state_compose, Phi, S, R.double(), out, stream=0, match="R is torch")


def test_kda(gdn):
    Hk, Hv, D, T = 2, 4, 64, 40
    td = torch.bfloat16
    cu = torch.tensor([0, 15, T], dtype=torch.int32)
    N = 2
    s = gdn.make_shape(Hk, Hv, D, D, N, 0, T, "bf16")
    qkv = torch.zeros(T, 2 * Hk * D + Hv * D, dtype=td)
    q, k, v = qkv[:, :Hk * D], qkv[:, Hk * D:2 * Hk * D], qkv[:, 2 * Hk * D:]
    alpha, beta = torch.zeros(T, Hv * D), torch.zeros(T, Hv)
    a_log, b_alpha = torch.zeros(Hv), torch.zeros(Hv * D)
    S, o = torch.zeros(N, Hv, D, D), torch.zeros(T, Hv * D, dtype=td)
    fwd = lambda **kw: gdn.gdn_kda_forward(
        s, q, k, v, kw.get("alpha", alpha), beta, a_log, kw.get("b_alpha", b_alpha), cu, S, S,
        o, stream=0)
    _fails(fwd, match=ON_DEVICE)
    _fails(fwd, alpha=torch.zeros(T, Hv), match="alpha is")            # one gate per channel
    _fails(fwd, b_alpha=torch.zeros(Hv), match="b_alpha has")
    dqkv = torch.zeros_like(qkv)
    ws = torch.zeros(gdn.gdn_kda_backward_workspace_bytes(s), dtype=torch.uint8)
    bwd = lambda **kw: gdn.gdn_kda_backward(
        s, q, k, v, alpha, beta, a_log, b_alpha, cu, S, o, S, dqkv[:, :Hk * D],
        dqkv[:, Hk * D:2 * Hk * D], dqkv[:, 2 * Hk * D:], kw.get("dalpha", torch.zeros(T, Hv * D)),
        torch.zeros(T, Hv), torch.zeros(Hv), kw.get("db_alpha", torch.zeros(Hv * D)),
        torch.zeros(N, Hv, D, D), ws, stream=0)
    _fails(bwd, match=ON_DEVICE)
    _fails(bwd, dalpha=torch.zeros(T, Hv), match="dalpha is")
    _fails(bwd, db_alpha=torch.zeros(Hv * D - 1), match="db_alpha has")


def test_device_status_needs_a_device_workspace(gdn):
    _fails(gdn.gdn_read_device_status, torch.zeros(256, dtype=torch.uint8), stream=0,
           match=ON_DEVICE)
