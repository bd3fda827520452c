"""The KDA variant (a decay gate per key channel) on the GPU against the oracle's KDA
recurrence: decode steps (one-token sequences), varlen prefills in token form (empty,
one-token and multi-chunk sequences), in-place state, the modulo head map, and the
reduction to the scalar gate against gdn_forward."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def _dev(torch, a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt or torch.float32)


def _case(dtype, Hk, Hv, Dk, Dv, seqlens, head_map=0, seed=3):
    wl = W.custom(dtype=dtype, seed=seed, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=seqlens,
                  S0_std=0.3, dt_bias_std=0.3, packed=False, head_map=head_map)
    inp = W.generate(wl)
    alpha, b_alpha = W.generate_kda_gates(wl)
    return wl, inp, alpha, b_alpha


def _run(torch, gdn, wl, inp, alpha, b_alpha, in_place=False):
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T, N = wl.total_tokens, len(inp.cu_seqlens) - 1
    q, k, v = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v))
    S_in = None if inp.S0 is None else _dev(torch, inp.S0)
    S_out = S_in if in_place else torch.full((N, wl.Hv, wl.Dk, wl.Dv), float("nan"),
                                              device="cuda")
    o = torch.full((T, wl.Hv * wl.Dv), float("nan"), device="cuda", dtype=td)
    shape = gdn.make_shape(wl.Hk, wl.Hv, wl.Dk, wl.Dv, N, 0, T, wl.dtype, wl.scale_value(),
                           wl.head_map)
    gdn.gdn_kda_forward(shape, q, k, v, _dev(torch, alpha), _dev(torch, inp.beta_raw),
                        _dev(torch, inp.a_log), _dev(torch, b_alpha),
                        _dev(torch, inp.cu_seqlens, torch.int32), S_in, S_out, o)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S_out.cpu().numpy()


def _ref(wl, inp, alpha, b_alpha):
    return oracle.kda_forward(inp.q, inp.k, inp.v, alpha, inp.beta_raw, inp.a_log, b_alpha,
                              inp.cu_seqlens, inp.S0, Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv,
                              scale=wl.scale_value(), head_map=wl.head_map)


@pytest.mark.parametrize("dtype,Hk,Hv,Dk,Dv,seqlens", [
    ("f32", 2, 6, 64, 32, (1,) * 7),              # decode: one token per sequence
    ("bf16", 2, 6, 128, 128, (1,) * 5),
    ("f32", 1, 2, 16, 16, (70, 1, 0, 130)),       # prefill: varlen, empty, one-token
    ("bf16", 2, 4, 128, 64, (200, 57)),
    ("bf16", 4, 4, 32, 128, (90,)),
])
def test_matches_the_oracle(dtype, Hk, Hv, Dk, Dv, seqlens):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha = _case(dtype, Hk, Hv, Dk, Dv, seqlens)
    o, S_T = _run(torch, gdn, wl, inp, alpha, b_alpha)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(S_T, S_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place_state_and_modulo_head_map(dtype):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha = _case(dtype, 2, 6, 64, 64, (33, 5), head_map=1, seed=8)
    o, S_T = _run(torch, gdn, wl, inp, alpha, b_alpha, in_place=True)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha)
    assert rel_err(o, o_ref) <= TOL[dtype]
    assert rel_err(S_T, S_ref) <= TOL[dtype]


def test_equal_channel_gates_match_the_scalar_gate_path():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, _, _ = _case("f32", 2, 4, 64, 64, (150, 40), seed=12)
    Dk = wl.Dk
    alpha = np.repeat(inp.alpha, Dk, axis=1)
    b_alpha = np.repeat(inp.dt_bias, Dk)
    o, S_T = _run(torch, gdn, wl, inp, alpha, b_alpha)
    layer = gdn.Layer.create(wl.Hk, wl.Hv, Dk, wl.Dv, inp.cu_seqlens, "f32", wl.scale_value())
    q, k, v = (_dev(torch, x) for x in (inp.q, inp.k, inp.v))
    o2 = torch.empty_like(v)
    S2 = torch.empty(2, wl.Hv, Dk, wl.Dv, device="cuda")
    layer.forward(q, k, v, _dev(torch, inp.alpha), _dev(torch, inp.beta_raw),
                  _dev(torch, inp.a_log), _dev(torch, inp.dt_bias), _dev(torch, inp.S0), o2, S2,
                  keep_states=False)
    torch.cuda.synchronize()
    assert rel_err(o, o2.cpu().numpy()) <= TOL["f32"]
    assert rel_err(S_T, S2.cpu().numpy()) <= TOL["f32"]


def test_rejects_bad_arguments():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    N, D, Hv = 2, 32, 2
    z = lambda *s: torch.zeros(*s, device="cuda")
    shape = gdn.make_shape(1, Hv, D, D, N, 0, N, "f32", 0.0)
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    q, v = z(N, D), z(N, Hv * D)
    with pytest.raises(gdn.GdnError):     # alpha narrower than Hv*Dk
        gdn.gdn_kda_forward(shape, q, q, v, z(N, Hv), z(N, Hv), z(Hv), z(Hv * D), cu, None,
                            z(N, Hv, D, D), v.clone())
    with pytest.raises(gdn.GdnError):     # no cu_seqlens
        gdn.gdn_kda_forward(shape, q, q, v, z(N, Hv * D), z(N, Hv), z(Hv), z(Hv * D), None, None,
                            z(N, Hv, D, D), v.clone())


@pytest.mark.slow
def test_full_layer_prefill_against_the_oracle_on_every_element():
    """The 27B-shaped layer (4096 tokens, 16 key / 48 value heads of 128, bf16) as one KDA
    prefill in token form."""
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    base = W.get("l27b_bf16")
    wl = W.custom(dtype="bf16", seed=base.seed, Hk=base.Hk, Hv=base.Hv, Dk=base.Dk, Dv=base.Dv,
                  seqlens=base.seqlens, S0_std=0.1, dt_bias_std=0.3, packed=True)
    inp = W.generate(wl)
    alpha, b_alpha = W.generate_kda_gates(wl)
    o, S_T = _run(torch, gdn, wl, inp, alpha, b_alpha)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(S_T, S_ref) <= TOL["bf16"]


def _run_bwd(torch, gdn, wl, inp, alpha, b_alpha, dS_T):
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T, N = wl.total_tokens, len(inp.cu_seqlens) - 1
    Hk, Hv, Dk, Dv = wl.Hk, wl.Hv, wl.Dk, wl.Dv
    q, k, v, dO = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v, inp.dO))
    nan = lambda *s, dt=torch.float32: torch.full(s, float("nan"), device="cuda", dtype=dt)
    g = dict(dq=nan(T, Hk * Dk, dt=td), dk=nan(T, Hk * Dk, dt=td), dv=nan(T, Hv * Dv, dt=td),
             dalpha=nan(T, Hv * Dk), dbeta_raw=nan(T, Hv), da_log=nan(Hv), db_alpha=nan(Hv * Dk),
             dS0=nan(N, Hv, Dk, Dv))
    shape = gdn.make_shape(Hk, Hv, Dk, Dv, N, 0, T, wl.dtype, wl.scale_value(), wl.head_map)
    ws = torch.empty(gdn.gdn_kda_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    gdn.gdn_kda_backward(shape, q, k, v, _dev(torch, alpha), _dev(torch, inp.beta_raw),
                         _dev(torch, inp.a_log), _dev(torch, b_alpha),
                         _dev(torch, inp.cu_seqlens, torch.int32),
                         None if inp.S0 is None else _dev(torch, inp.S0), dO,
                         None if dS_T is None else _dev(torch, dS_T), g["dq"], g["dk"], g["dv"],
                         g["dalpha"], g["dbeta_raw"], g["da_log"], g["db_alpha"], g["dS0"], ws)
    torch.cuda.synchronize()
    return {key: val.float().cpu().numpy() for key, val in g.items()}


@pytest.mark.parametrize("dtype,Hk,Hv,Dk,Dv,seqlens,head_map", [
    ("f32", 1, 2, 16, 32, (1, 9, 0, 20), 0),      # segments of 8: ragged, empty, one-token
    ("f32", 2, 4, 64, 64, (37, 70), 0),
    ("bf16", 2, 6, 128, 128, (45, 18), 0),
    ("bf16", 2, 4, 32, 64, (33,), 1),              # modulo head map
])
def test_backward_matches_the_oracle(dtype, Hk, Hv, Dk, Dv, seqlens, head_map):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha = _case(dtype, Hk, Hv, Dk, Dv, seqlens, head_map=head_map, seed=17)
    dS_T = (0.3 * np.random.default_rng(4).standard_normal(inp.S0.shape)).astype(np.float32)
    got = _run_bwd(torch, gdn, wl, inp, alpha, b_alpha, dS_T)
    ref = oracle.kda_backward(inp.q, inp.k, inp.v, alpha, inp.beta_raw, inp.a_log, b_alpha,
                              inp.cu_seqlens, inp.dO, inp.S0, dS_T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv,
                              scale=wl.scale_value(), head_map=head_map)
    for key in ("dq", "dk", "dv", "dalpha", "dbeta_raw", "da_log", "db_alpha", "dS0"):
        assert rel_err(got[key], ref[key]) <= TOL[dtype], key


def test_backward_is_bit_reproducible():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha = _case("bf16", 2, 4, 64, 64, (50, 31), seed=19)
    a = _run_bwd(torch, gdn, wl, inp, alpha, b_alpha, None)
    b = _run_bwd(torch, gdn, wl, inp, alpha, b_alpha, None)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.slow
def test_backward_at_the_full_head_shape():
    """16 key heads shared by 48 value heads of 128, bf16, two sequences (256 tokens: the
    oracle's KDA backward keeps every state)."""
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha = _case("bf16", 16, 48, 128, 128, (100, 156), seed=23)
    dS_T = (0.1 * np.random.default_rng(6).standard_normal(inp.S0.shape)).astype(np.float32)
    got = _run_bwd(torch, gdn, wl, inp, alpha, b_alpha, dS_T)
    ref = oracle.kda_backward(inp.q, inp.k, inp.v, alpha, inp.beta_raw, inp.a_log, b_alpha,
                              inp.cu_seqlens, inp.dO, inp.S0, dS_T, Hk=16, Hv=48, Dk=128, Dv=128,
                              scale=wl.scale_value())
    for key in ("dq", "dk", "dv", "dalpha", "dbeta_raw", "da_log", "db_alpha", "dS0"):
        assert rel_err(got[key], ref[key]) <= TOL["bf16"], key
