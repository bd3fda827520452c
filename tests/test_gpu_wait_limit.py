"""A bounded wait that runs out: the failure path of the fused forward's flag waits.

In the fused forward the chunk walks wait for the preparation units' readiness flags,
each wait bounded by GDN_FLAG_WAIT_LIMIT_NS of wall time, after which the walk records
GDN_ERR_TIMEOUT in the status word and carries on (it never spins without bound).  This
test builds a copy of the library whose flag waits give up at once (the limit set to 0),
runs a forward through it whose walks must wait (the first chunk's preparation takes
microseconds), and checks that the launch ends, that the status word says
GDN_ERR_TIMEOUT, and that the same process then runs a clean training step with the
regular library that matches the oracle.  Nothing faults, traps or hangs: the waits are
the same bounded loops, only their limit is shorter.
"""
import ctypes
import os
import tempfile

import pytest

import workloads as W
from tests.gdn_harness import DeviceRun, TOL, compare, oracle_outputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch


def _variant_library(path):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "gdn_build", os.path.join(ROOT, "gated_deltanet_backward_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build_variant(path, {"GDN_FLAG_WAIT_LIMIT_NS": 0}, sources=("gdn_tc_fwd.cu",))


def test_flag_wait_that_runs_out_records_timeout_and_the_process_goes_on(torch_cuda,
                                                                        monkeypatch):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    # one sequence, 12 walks: the forward runs as one fused launch (walks + preparation)
    wl = W.custom(dtype="bf16", Hk=4, Hv=12, Dk=128, Dv=128, seqlens=(2048,), seed=21,
                  S0_std=0.1, dST_std=0.01, dt_bias_std=0.1)
    inp = W.generate(wl)
    with tempfile.TemporaryDirectory() as tmp:
        lib = ctypes.CDLL(_variant_library(os.path.join(tmp, "libgdn_flagwait0.so")))
        for name in ("gdn_forward", "gdn_read_device_status", "gdn_status_string",
                     "gdn_last_error", "gdn_workspace_bytes", "gdn_saved_state_bytes"):
            getattr(lib, name).argtypes = getattr(gdn._lib, name).argtypes
            getattr(lib, name).restype = getattr(gdn._lib, name).restype
        run = DeviceRun(inp, run_backward=False, train=False)   # buffers (regular library)
        o = torch.zeros_like(run.o)
        S_T = torch.zeros_like(run.S_T)
        with monkeypatch.context() as m:
            m.setattr(gdn, "_lib", lib)
            gdn.gdn_forward(run.layer.shape, run.q, run.k, run.v, run.alpha, run.beta_raw,
                            run.a_log, run.dt_bias, run.layer.cu_seqlens,
                            run.layer.chunk_offsets, run.S0, o, S_T, run.layer.saved_states,
                            run.layer.ws_fwd)
            status = gdn.gdn_read_device_status(run.layer.ws_fwd)   # synchronises
        torch.cuda.synchronize()
        assert status == -5, gdn.gdn_status_string(status)          # GDN_ERR_TIMEOUT
    # the context is intact: a clean training step with the regular library
    clean = DeviceRun(inp)
    assert clean.status() == 0 and clean.status(backward=True) == 0
    compare(clean.host(), oracle_outputs(inp), TOL["bf16"])
