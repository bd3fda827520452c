"""The forward with the gated RMSNorm of its output fused in (gdn_forward_gated_rmsnorm),
on the GPU against the oracle's composition forward -> gated RMSNorm and against the
library's own unfused pair gdn_forward -> gdn_gated_rmsnorm_forward.

* o is bit-identical to gdn_forward's on the same inputs (the norm only reads it);
* y matches the oracle's composition within the path's tolerance, on ragged varlen
  batches (several chunks, a ragged tail, an empty sequence), every value-head size,
  strided row views of z and y, and both dtypes;
* y matches the unfused norm of the same o to within a bf16 rounding step (the fused
  epilogue sums the row's squares in another order), and exactly for fp32, where the
  fused entry point runs the same norm kernel;
* a keeping (training) forward through the fused entry point feeds the backward as
  gdn_forward's does: the same gradients bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, DeviceRun, oracle_outputs, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch


def _case(dtype, Hk, Hv, D, seqlens, seed):
    wl = W.custom(dtype=dtype, Hk=Hk, Hv=Hv, Dk=D, Dv=D, seqlens=seqlens, seed=seed,
                  S0_std=0.1, dST_std=0.01, dt_bias_std=0.1)
    return W.generate(wl), W.generate_layer_steps(wl)


def _fused(torch, gdn, run, ls, eps, pad):
    """gdn_forward_gated_rmsnorm on run's inputs into fresh o / y (z, y strided by pad)."""
    T, Wd = run.o.shape
    td = run.o.dtype

    def view(a):
        buf = torch.zeros((T, Wd + pad), device="cuda", dtype=td)
        buf[:, :Wd] = torch.from_numpy(np.ascontiguousarray(a)).to("cuda", td)
        return buf[:, :Wd]

    z = view(ls.z)
    y = torch.full((T, Wd + pad), float("nan"), device="cuda", dtype=td)[:, :Wd]
    o = torch.full_like(run.o, float("nan"))
    S_T = torch.full_like(run.S_T, float("nan"))
    gamma = torch.from_numpy(ls.gamma).cuda()
    L = run.layer
    gdn.gdn_forward_gated_rmsnorm(L.shape, run.q, run.k, run.v, run.alpha, run.beta_raw,
                                  run.a_log, run.dt_bias, L.cu_seqlens, L.chunk_offsets,
                                  run.S0, o, S_T, L.saved_states, z, gamma, eps, y, L.ws_fwd)
    status = gdn.gdn_read_device_status(L.ws_fwd)
    assert status == 0, gdn.gdn_status_string(status)
    return o, S_T, z, gamma, y


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D,Hk,Hv,seqlens,eps,pad", [
    (128, 2, 6, (300, 0, 77, 129), 1e-6, 0),
    (64, 1, 3, (200, 64), 1e-5, 8),
    (32, 2, 2, (150,), 0.25, 0),
    (16, 1, 4, (65, 3), 1e-6, 8),
])
def test_fused_norm_matches_the_oracle_and_the_unfused_pair(torch_cuda, dtype, D, Hk, Hv,
                                                            seqlens, eps, pad):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    inp, ls = _case(dtype, Hk, Hv, D, seqlens, seed=D + Hv)
    run = DeviceRun(inp, run_backward=False, train=False)   # gdn_forward's o
    o, S_T, z, gamma, y = _fused(torch, gdn, run, ls, eps, pad)
    y_unfused = torch.full_like(y, float("nan"))
    gdn.gdn_gated_rmsnorm_forward(o, z, gamma, y_unfused, eps)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy()
    assert np.array_equal(f(o), f(run.o))
    assert np.array_equal(f(S_T), f(run.S_T))
    yf, yu = f(y), f(y_unfused)
    assert np.all(np.isfinite(yf))
    if dtype == "f32":
        assert np.array_equal(yf, yu)
    else:
        # one bf16 rounding step (2^-8 relative) either way, plus the fp32 sums' own order
        assert np.all(np.abs(yf - yu) <= 2.0 ** -7 * np.abs(yu) + 1e-6)
    o_ref = oracle_outputs(inp, backward=False)["o"]
    y_ref = oracle.gated_rmsnorm_forward(o_ref, ls.z, ls.gamma, Hv, D, eps)
    assert rel_err(yf, y_ref) <= TOL[dtype]


def test_fused_norm_training_forward_feeds_the_backward_unchanged(torch_cuda):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    inp, ls = _case("bf16", 2, 4, 128, (260, 100), seed=5)
    plain = DeviceRun(inp)                    # gdn_forward + gdn_backward, training step
    fused = DeviceRun(inp, run_backward=False)
    L = fused.layer
    z = torch.from_numpy(ls.z).to("cuda", torch.bfloat16)
    gamma = torch.from_numpy(ls.gamma).cuda()
    y = torch.empty_like(z)
    fused.o.fill_(float("nan"))
    L.saved_states.zero_()
    gdn.gdn_forward_gated_rmsnorm(L.shape, fused.q, fused.k, fused.v, fused.alpha,
                                  fused.beta_raw, fused.a_log, fused.dt_bias, L.cu_seqlens,
                                  L.chunk_offsets, fused.S0, fused.o, fused.S_T, L.saved_states, z,
                                  gamma, 1e-6, y, L.ws_bwd,
                                  flags=gdn.GDN_FLAG_KEEP_FOR_BACKWARD)
    fused.run_backward()
    a, b = plain.host(), fused.host()
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
