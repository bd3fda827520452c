"""gdn_decode_step on the GPU against the oracle's token-by-token forward.

A decode step is the recurrence applied once per sequence, so N sequences of one token
each through the oracle's forward give its exact o and S_T; T steps fed one token row at
a time must reproduce the forward over sequences of T tokens (the last state and every
output row)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def _dev(torch, a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda",
                                                        dtype=dt or torch.float32)


def _oracle_forward(inp):
    wl = inp.wl
    return oracle.forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                          inp.cu_seqlens, inp.S0, Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv,
                          scale=wl.scale_value())


@pytest.mark.parametrize("dtype,Hk,Hv,Dk,Dv,N,S0_std", [
    ("f32", 2, 6, 64, 32, 5, 0.3),
    ("bf16", 2, 6, 128, 64, 7, 0.3),
    ("bf16", 4, 4, 32, 128, 3, 0.0),     # zero state (S_in = NULL)
    ("f32", 1, 2, 16, 16, 1, 0.5),
])
def test_one_step_matches_the_token_recurrence(dtype, Hk, Hv, Dk, Dv, N, S0_std):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl = W.custom(dtype=dtype, seed=21, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=(1,) * N,
                  S0_std=S0_std, dt_bias_std=0.2, packed=False)
    inp = W.generate(wl)
    o_ref, S_ref = _oracle_forward(inp)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v))
    alpha, beta_raw = _dev(torch, inp.alpha), _dev(torch, inp.beta_raw)
    a_log, dt_bias = _dev(torch, inp.a_log), _dev(torch, inp.dt_bias)
    S_in = None if inp.S0 is None else _dev(torch, inp.S0)
    S_out = torch.full((N, Hv, Dk, Dv), float("nan"), device="cuda")
    o = torch.full((N, Hv * Dv), float("nan"), device="cuda", dtype=td)
    shape = gdn.make_shape(Hk, Hv, Dk, Dv, N, N, N, dtype, wl.scale_value())
    gdn.gdn_decode_step(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, S_in, S_out, o)
    torch.cuda.synchronize()
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL[dtype]
    assert rel_err(S_out.cpu().numpy(), S_ref) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_steps_in_place_reproduce_the_forward(dtype):
    """Three steps updating the state in place (S_out = S_in) equal the forward over
    sequences of three tokens: every output row and the final state."""
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    N, T, Hk, Hv, Dk, Dv = 4, 3, 2, 4, 64, 64
    wl = W.custom(dtype=dtype, seed=5, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=(T,) * N,
                  S0_std=0.3, dt_bias_std=0.2, packed=False)
    inp = W.generate(wl)
    o_ref, S_ref = _oracle_forward(inp)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    shape = gdn.make_shape(Hk, Hv, Dk, Dv, N, N, N, dtype, wl.scale_value())
    S = _dev(torch, inp.S0)
    a_log, dt_bias = _dev(torch, inp.a_log), _dev(torch, inp.dt_bias)
    o_rows = np.zeros_like(o_ref)
    for t in range(T):
        rows = np.arange(N) * T + t          # token t of every sequence
        q, k, v = (_dev(torch, x[rows], td) for x in (inp.q, inp.k, inp.v))
        alpha, beta_raw = _dev(torch, inp.alpha[rows]), _dev(torch, inp.beta_raw[rows])
        o = torch.full((N, Hv * Dv), float("nan"), device="cuda", dtype=td)
        gdn.gdn_decode_step(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, S, S, o)
        o_rows[rows] = o.float().cpu().numpy()
    torch.cuda.synchronize()
    assert rel_err(o_rows, o_ref) <= TOL[dtype]
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL["f32"]


def test_rejects_bad_arguments_before_launching():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    N, Hk, Hv, D = 2, 1, 2, 32
    shape = gdn.make_shape(Hk, Hv, D, D, N, N, N, "f32", 0.0)
    z = lambda *s: torch.zeros(*s, device="cuda")
    q, k, v, o = z(N, D), z(N, D), z(N, Hv * D), z(N, Hv * D)
    g, a = z(N, Hv), z(Hv)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_decode_step(shape, q, k, v, g, g, a, a, None, None, o)   # no S_out
    bad = gdn.make_shape(Hk, Hv, 24, D, N, N, N, "f32", 0.0)             # unsupported Dk
    with pytest.raises(gdn.GdnError):
        gdn.gdn_decode_step(bad, q, k, v, g, g, a, a, None, z(N, Hv, 24, D), o)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_step_with_the_modulo_head_map(dtype):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    N, Hk, Hv, Dk, Dv = 3, 2, 6, 64, 32
    wl = W.custom(dtype=dtype, seed=23, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=(1,) * N,
                  S0_std=0.3, dt_bias_std=0.2, packed=False, head_map=1)
    inp = W.generate(wl)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log,
                                  inp.dt_bias, inp.cu_seqlens, inp.S0, Hk=Hk, Hv=Hv, Dk=Dk,
                                  Dv=Dv, scale=wl.scale_value(), head_map=1)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v))
    S = _dev(torch, inp.S0)
    o = torch.full((N, Hv * Dv), float("nan"), device="cuda", dtype=td)
    shape = gdn.make_shape(Hk, Hv, Dk, Dv, N, N, N, dtype, wl.scale_value(),
                           gdn.GDN_HEAD_MAP_MODULO)
    gdn.gdn_decode_step(shape, q, k, v, _dev(torch, inp.alpha), _dev(torch, inp.beta_raw),
                        _dev(torch, inp.a_log), _dev(torch, inp.dt_bias), S, S, o)
    torch.cuda.synchronize()
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL[dtype]
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL["f32"]
