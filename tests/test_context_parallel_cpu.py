"""Context parallelism's host logic on the CPU: the orchestration of
gated_deltanet_backward_gb300.context_parallel (segment maps, exchange, scans, final
passes, the all-reduce of the shared-parameter gradients) driven by an oracle backend,
in one process and as two or four gloo ranks, against the oracle run over the whole
sequence.
The CUDA backend is checked on the GPU (tests/test_gpu_context.py)."""
import os
import socket
import sys

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")


def _cp():
    # the orchestration module only: importing the package itself loads the CUDA library
    import importlib.util
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = os.path.join(here, "gated_deltanet_backward_gb300", "context_parallel.py")
    spec = importlib.util.spec_from_file_location("gdn_context_parallel", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # dataclasses resolve annotations through it
    spec.loader.exec_module(mod)
    return mod


class OracleSegmentOps:
    """The steps of one segment through the oracle (f64, CPU tensors)."""

    def __init__(self, Hk, Hv, Dk, Dv, scale):
        self.kw = dict(Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, scale=scale)
        self.Hv, self.Dk, self.Dv = Hv, Dk, Dv

    @staticmethod
    def _cu(seg):
        return np.array([0, seg.q.shape[0]], np.int32)

    @staticmethod
    def _np(t):
        return None if t is None else t.numpy()

    def zero_state(self):
        return torch.zeros(1, self.Hv, self.Dk, self.Dv, dtype=torch.float64)

    def state_map(self, seg):
        n = self._np
        Phi = oracle.state_map(n(seg.q), n(seg.k), n(seg.alpha), n(seg.beta_raw), n(seg.a_log),
                               n(seg.dt_bias), self._cu(seg), Hk=self.kw["Hk"], Hv=self.Hv,
                               Dk=self.Dk)
        return torch.from_numpy(Phi)

    def forward(self, seg, S_in, keep):
        n = self._np
        o, S_T = oracle.forward(n(seg.q), n(seg.k), n(seg.v), n(seg.alpha), n(seg.beta_raw),
                                n(seg.a_log), n(seg.dt_bias), self._cu(seg), n(S_in), **self.kw)
        return torch.from_numpy(o), torch.from_numpy(S_T)

    def backward(self, seg, S_in, dO, dS_out):
        n = self._np
        g = oracle.backward(n(seg.q), n(seg.k), n(seg.v), n(seg.alpha), n(seg.beta_raw),
                            n(seg.a_log), n(seg.dt_bias), self._cu(seg), n(dO), n(S_in),
                            n(dS_out), **self.kw)
        return {k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in g.items()}

    def compose(self, Phi, S, R, transpose):
        P = Phi.transpose(-1, -2) if transpose else Phi
        return torch.matmul(P, S) + R


def _problem(seed=11, L=(23, 9, 31, 17)):
    wl = W.custom(Hk=2, Hv=4, Dk=8, Dv=6, seqlens=(sum(L),), S0_std=0.4, dt_bias_std=0.3,
                  packed=False, seed=seed)
    inp = W.generate(wl)
    rng = np.random.default_rng(seed)
    dS_T = rng.standard_normal(inp.S0.shape)
    return wl, inp, dS_T, L


def _whole(wl, inp, dS_T):
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, scale=wl.scale_value())
    o, S_T = oracle.forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                            inp.cu_seqlens, inp.S0, **kw)
    g = oracle.backward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                        inp.cu_seqlens, inp.dO, inp.S0, dS_T, **kw)
    return o, S_T, g


def _segments(cp, inp, L, which):
    bounds = np.concatenate([[0], np.cumsum(L)])
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    segs = []
    for s in which:
        r = slice(bounds[s], bounds[s + 1])
        segs.append(cp.Segment(f(inp.q[r]), f(inp.k[r]), f(inp.v[r]), f(inp.alpha[r]),
                               f(inp.beta_raw[r]), f(inp.a_log), f(inp.dt_bias)))
    return segs, bounds


def _run_and_check(cp, group, which, wl, inp, dS_T, L):
    ops = OracleSegmentOps(wl.Hk, wl.Hv, wl.Dk, wl.Dv, wl.scale_value())
    segs, bounds = _segments(cp, inp, L, which)
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    outs, S_T, ctx = cp.forward(ops, segs, f(inp.S0), group)
    dOs = [f(inp.dO[bounds[s]:bounds[s + 1]]) for s in which]
    grads, da_log, ddt, dS0 = cp.backward(ops, segs, ctx, dOs, f(dS_T), group)
    o_ref, S_ref, g_ref = _whole(wl, inp, dS_T)
    tol = dict(rtol=0, atol=1e-10)
    assert np.allclose(S_T.numpy(), S_ref, **tol)
    for j, s in enumerate(which):
        r = slice(bounds[s], bounds[s + 1])
        assert np.allclose(outs[j].numpy(), o_ref[r], **tol)
        for key, ref in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dalpha", "dalpha"),
                         ("dbeta_raw", "dbeta_raw")):
            assert np.allclose(grads[j][key].numpy(), g_ref[ref][r], **tol), key
    assert np.allclose(da_log.numpy(), g_ref["da_log"], **tol)
    assert np.allclose(ddt.numpy(), g_ref["ddt_bias"], **tol)
    if which[0] == 0:
        assert np.allclose(dS0.numpy(), g_ref["dS0"], **tol)


def test_segments_in_one_process_equal_the_whole_sequence():
    cp = _cp()
    wl, inp, dS_T, L = _problem()
    _run_and_check(cp, cp.LocalGroup(), list(range(len(L))), wl, inp, dS_T, L)


def _rank_main(rank, world, port):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        cp = _cp()
        wl, inp, dS_T, L = _problem()
        per = len(L) // world
        _run_and_check(cp, cp.TorchGroup(), list(range(rank * per, rank * per + per)), wl, inp,
                       dS_T, L)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_holding_consecutive_segments_equal_the_whole_sequence(world):
    """Two ranks with two segments each, and four ranks with one segment each."""
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(world, _free_port()), nprocs=world, join=True)
