"""gdn_forward_noalloc: the forward for callers that cannot allocate device memory.

Callers that may not call cudaMalloc (a device-memory budget fixed at start-up,
a plugin host that passes only inputs and outputs, a path that cannot take the
implicit synchronisation of cudaMalloc / cudaFree) use this entry point; it runs
the forward with the library's built-in 64 MiB scratch array instead of a caller
workspace.  These tests call it through the C ABI twice in a row and compare
every output with the regular gdn_forward (same tolerance as the parity tests, and
bit for bit, since both run the same kernels),
and check that a shape needing more scratch is refused before any launch.

This file sorts last so that a run stopping at its first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import workloads as W
from tests.gdn_harness import DeviceRun, TOL, rel_err, saved_states_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch


@pytest.mark.parametrize("wl", [
    W.get("shared_kh_f32"),
    W.custom(dtype="bf16", Hk=2, Hv=6, Dk=128, Dv=128, seqlens=(300, 0, 77), seed=13,
             S0_std=0.1, dt_bias_std=0.1),
], ids=["shared_kh_f32", "bf16_varlen"])
def test_noalloc_forward_matches_the_workspace_forward(torch_cuda, wl):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    inp = W.generate(wl)
    # gdn_forward with a caller workspace and no flags: the same kernels as the no-alloc call
    run = DeviceRun(inp, run_backward=False, train=False)
    ref = run.host()
    nsaved = wl.total_chunks * wl.Hv * wl.Dk * wl.Dv
    for call in range(2):
        o = torch.full_like(run.o, float("nan"))
        S_T = torch.full_like(run.S_T, float("nan"))
        saved = torch.full((max(1, nsaved),), float("nan"), device="cuda")
        rc = gdn._lib.gdn_forward_noalloc(
            gdn.ctypes.byref(run.layer.shape), *gdn._mat(run.q), *gdn._mat(run.k),
            *gdn._mat(run.v), *gdn._mat(run.alpha), *gdn._mat(run.beta_raw),
            run.a_log.data_ptr(), run.dt_bias.data_ptr(), run.layer.cu_seqlens.data_ptr(),
            run.layer.chunk_offsets.data_ptr(), None if run.S0 is None else run.S0.data_ptr(),
            *gdn._mat(o), S_T.data_ptr(), saved.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert rc == 0, (call, gdn.gdn_status_string(rc), gdn.gdn_last_error())
        torch.cuda.synchronize()
        got = dict(o=o.double().cpu().numpy(), S_T=S_T.double().cpu().numpy(),
                   saved=saved_states_dense(saved, wl))
        for key in got:
            assert np.all(np.isfinite(got[key])), (call, key)
            assert rel_err(got[key], ref[key]) <= TOL[wl.dtype], (call, key)
            # both calls run the same kernels on the same inputs: the same bits
            assert np.array_equal(got[key], ref[key]), (call, key)


def test_noalloc_refuses_shapes_beyond_its_scratch(torch_cuda):
    import gated_deltanet_backward_gb300 as gdn
    # the 27B-shaped layer needs ~258 MB of forward scratch, above the 64 MiB built in
    shape = gdn.make_shape(16, 48, 128, 128, 1, 64, 4096, "bf16")
    assert gdn.gdn_workspace_bytes(shape, False) > 64 << 20
    with pytest.raises(gdn.GdnError) as err:
        gdn.gdn_forward_noalloc(shape, *([None] * 13), stream=0)
    assert err.value.code == -6
    assert "scratch" in gdn.gdn_last_error()
