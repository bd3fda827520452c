"""Context parallelism on the GPU: gdn_state_compose against the product it defines
(numpy, f64), and one sequence cut into segments -- the segment maps from gdn_forward,
the scans in gdn_state_compose, the final passes -- against the oracle run over the
whole sequence: every output row, the final state and every gradient."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def _dev(torch, a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt or torch.float32)


@pytest.mark.parametrize("n,Dk,Dv", [(5, 128, 64), (3, 16, 16), (2, 100, 72), (48, 128, 128)])
@pytest.mark.parametrize("transpose", [False, True])
def test_compose_matches_the_product(n, Dk, Dv, transpose):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    rng = np.random.default_rng(n + Dk)
    Phi = rng.standard_normal((n, Dk, Dk)).astype(np.float32)
    S = rng.standard_normal((n, Dk, Dv)).astype(np.float32)
    R = rng.standard_normal((n, Dk, Dv)).astype(np.float32)
    P = np.swapaxes(Phi, 1, 2) if transpose else Phi
    want = np.einsum("bij,bjk->bik", P.astype(np.float64), S.astype(np.float64)) + R
    dP, dS, dR = _dev(torch, Phi), _dev(torch, S), _dev(torch, R)
    out = torch.full_like(dR, float("nan"))
    gdn.gdn_state_compose(dP, dS, dR, out, transpose)
    gdn.gdn_state_compose(dP, dS, dR, dR, transpose)          # in place on R
    z = torch.full_like(dR, float("nan"))
    gdn.gdn_state_compose(dP, dS, None, z, transpose)         # R = 0
    torch.cuda.synchronize()
    assert rel_err(out.cpu().numpy(), want) <= 1e-5
    assert np.array_equal(dR.cpu().numpy(), out.cpu().numpy())
    assert rel_err(z.cpu().numpy(), want - R) <= 1e-5


def test_compose_rejects_overlap():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    a = torch.zeros(2, 16, 16, device="cuda")
    with pytest.raises(gdn.GdnError):
        gdn.gdn_state_compose(a, a.clone(), None, a)


@pytest.mark.parametrize("dtype,L", [("f32", (300, 100, 257)), ("bf16", (320, 64, 321)),
                                     ("bf16", (1000, 1000))])
def test_segments_equal_the_whole_sequence(dtype, L):
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    from gated_deltanet_backward_gb300 import context_parallel as cp
    Hk, Hv, D = 2, 4, 64
    wl = W.custom(dtype=dtype, seed=41, Hk=Hk, Hv=Hv, Dk=D, Dv=D, seqlens=(sum(L),),
                  S0_std=0.3, dt_bias_std=0.2, packed=False)
    inp = W.generate(wl)
    rng = np.random.default_rng(2)
    dS_T = (0.5 * rng.standard_normal(inp.S0.shape)).astype(np.float32)
    kw = dict(Hk=Hk, Hv=Hv, Dk=D, Dv=D, scale=wl.scale_value())
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log,
                                  inp.dt_bias, inp.cu_seqlens, inp.S0, **kw)
    g_ref = oracle.backward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                            inp.cu_seqlens, inp.dO, inp.S0, dS_T, **kw)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    bounds = np.concatenate([[0], np.cumsum(L)])
    segs, dOs = [], []
    a_log, dt_bias = _dev(torch, inp.a_log), _dev(torch, inp.dt_bias)
    for s in range(len(L)):
        r = slice(bounds[s], bounds[s + 1])
        segs.append(cp.Segment(_dev(torch, inp.q[r], td), _dev(torch, inp.k[r], td),
                               _dev(torch, inp.v[r], td), _dev(torch, inp.alpha[r]),
                               _dev(torch, inp.beta_raw[r]), a_log, dt_bias))
        dOs.append(_dev(torch, inp.dO[r], td))
    ops = cp.GpuSegmentOps(Hk, Hv, D, D, dtype, wl.scale_value())
    outs, S_T, ctx = cp.forward(ops, segs, _dev(torch, inp.S0))
    grads, da_log, ddt, dS0 = cp.backward(ops, segs, ctx, dOs, _dev(torch, dS_T))
    torch.cuda.synchronize()
    cat = lambda key: np.concatenate([g[key].float().cpu().numpy() for g in grads])
    tol = TOL[dtype]
    assert rel_err(np.concatenate([o.float().cpu().numpy() for o in outs]), o_ref) <= tol
    assert rel_err(S_T.cpu().numpy(), S_ref) <= tol
    for key in ("dq", "dk", "dv", "dalpha", "dbeta_raw"):
        assert rel_err(cat(key), g_ref[key]) <= tol, key
    assert rel_err(da_log.cpu().numpy(), g_ref["da_log"]) <= tol
    assert rel_err(ddt.cpu().numpy(), g_ref["ddt_bias"]) <= tol
    assert rel_err(dS0.cpu().numpy(), g_ref["dS0"]) <= tol
    assert gdn.gdn_read_device_status(segs[0].state["layer"].ws_bwd) == 0
