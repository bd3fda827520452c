"""Data-parallel sharding of one batch (gated_deltanet_backward_gb300.sharding) on the
CPU, as gloo ranks with the oracle computing each rank's shard:

* key-head groups: every rank runs its key heads and their value heads, with nothing
  exchanged; the gathered outputs equal the whole batch's oracle run bit for bit (the
  oracle's units are (sequence, key head), so a head subset computes the same sums in
  the same order);
* sequences: every rank runs its whole sequences; d a_log and d dt_bias are all-gathered
  and added in rank order; the per-token outputs and states equal the whole batch's bit
  for bit and the shared-parameter gradients to f64 rounding (the sum is regrouped).

The GPU library takes the same views (pointer offsets, row strides and a sub-shape)."""
import importlib.util
import os
import socket
import sys

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sharding():
    # the sharding module alone: importing the package loads the CUDA library
    path = os.path.join(ROOT, "gated_deltanet_backward_gb300", "sharding.py")
    spec = importlib.util.spec_from_file_location("gdn_sharding", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    return W.custom(Hk=4, Hv=12, Dk=8, Dv=6, seqlens=(37, 0, 64, 5, 90, 21), S0_std=0.3,
                    dST_std=0.2, dt_bias_std=0.3, seed=17)


def _oracle(inp, wl, cu, S0, dS_T, q, k, v, alpha, beta_raw, a_log, dt_bias, dO):
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, scale=wl.scale_value())
    o, S_T, states = oracle.forward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu, S0,
                                    chunk=W.CHUNK, **kw)
    g = oracle.backward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu, dO, S0, dS_T, **kw)
    return dict(o=o, S_T=S_T, saved=states, **g)


def _whole(inp):
    wl = inp.wl
    return _oracle(inp, wl, inp.cu_seqlens, inp.S0, inp.dS_T, inp.q, inp.k, inp.v, inp.alpha,
                   inp.beta_raw, inp.a_log, inp.dt_bias, inp.dO)


def _heads_rank(rank, world, port, out_q):
    import torch.distributed as dist
    sh_mod = _sharding()
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        inp = W.generate(_workload())
        wl = inp.wl
        sh = sh_mod.head_shard(wl.Hk, wl.Hv, world, rank)
        vw = sh_mod.shard_heads(sh, wl.Dk, wl.Dv, q=inp.q, k=inp.k, v=inp.v, alpha=inp.alpha,
                                beta_raw=inp.beta_raw, a_log=inp.a_log, dt_bias=inp.dt_bias,
                                dO=inp.dO)
        sub = W.replace(wl, Hk=sh.Hk, Hv=sh.Hv)
        hs = slice(sh.h0, sh.h1)
        res = _oracle(inp, sub, inp.cu_seqlens, inp.S0[:, hs], inp.dS_T[:, hs], vw["q"],
                      vw["k"], vw["v"], vw["alpha"], vw["beta_raw"], vw["a_log"], vw["dt_bias"],
                      vw["dO"])
        gathered = [None] * world
        dist.all_gather_object(gathered, (sh.h0, sh.h1, sh.kh0, sh.kh1, res))
        if rank == 0:
            out_q.put(gathered)
    finally:
        dist.destroy_process_group()


def _seq_rank(rank, world, port, out_q):
    import torch.distributed as dist
    sh_mod = _sharding()
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        inp = W.generate(_workload())
        wl = inp.wl
        sh = sh_mod.sequence_shard(inp.cu_seqlens, world, rank)
        vw = sh_mod.shard_sequences(sh, q=inp.q, k=inp.k, v=inp.v, alpha=inp.alpha,
                                    beta_raw=inp.beta_raw, a_log=inp.a_log,
                                    dt_bias=inp.dt_bias, dO=inp.dO, S0=inp.S0, dS_T=inp.dS_T)
        sub = W.replace(wl, seqlens=tuple(np.diff(sh.cu_seqlens).tolist()))
        res = _oracle(inp, sub, sh.cu_seqlens, vw["S0"], vw["dS_T"], vw["q"], vw["k"], vw["v"],
                      vw["alpha"], vw["beta_raw"], vw["a_log"], vw["dt_bias"], vw["dO"])
        da, dd = sh_mod.reduce_gate_grads(torch.from_numpy(res["da_log"]),
                                          torch.from_numpy(res["ddt_bias"]))
        res["da_log"], res["ddt_bias"] = da.numpy(), dd.numpy()
        gathered = [None] * world
        dist.all_gather_object(gathered, (sh.n0, sh.n1, sh.t0, sh.t1, res))
        if rank == 0:
            out_q.put(gathered)
    finally:
        dist.destroy_process_group()


def _spawn(fn, world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=fn, args=(r, world, _PORT[0], q)) for r in range(world)]
    for p in procs:
        p.start()
    out = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return out


_PORT = [0]


@pytest.mark.parametrize("world", [2, 4])
def test_key_head_shards_equal_the_whole_batch_bit_for_bit(world):
    _PORT[0] = _free_port()
    parts = _spawn(_heads_rank, world)
    inp = W.generate(_workload())
    whole = _whole(inp)
    wl = inp.wl
    seen = np.zeros(wl.Hv, bool)
    for h0, h1, kh0, kh1, res in parts:
        seen[h0:h1] = True
        cv, ck, hs = slice(h0 * wl.Dv, h1 * wl.Dv), slice(kh0 * wl.Dk, kh1 * wl.Dk), slice(h0, h1)
        for key, sl in (("o", (slice(None), cv)), ("dv", (slice(None), cv)),
                        ("dq", (slice(None), ck)), ("dk", (slice(None), ck)),
                        ("dalpha", (slice(None), hs)), ("dbeta_raw", (slice(None), hs)),
                        ("S_T", (slice(None), hs)), ("dS0", (slice(None), hs)),
                        ("saved", (slice(None), hs)), ("da_log", (hs,)), ("ddt_bias", (hs,))):
            assert np.array_equal(res[key], whole[key][sl]), (world, h0, key)
    assert seen.all()


def test_sequence_shards_equal_the_whole_batch():
    _PORT[0] = _free_port()
    world = 2
    parts = _spawn(_seq_rank, world)
    inp = W.generate(_workload())
    whole = _whole(inp)
    covered = 0
    chunk_off = oracle.chunk_offsets(inp.cu_seqlens, W.CHUNK)
    for n0, n1, t0, t1, res in parts:
        covered += t1 - t0
        rows = slice(t0, t1)
        for key in ("o", "dq", "dk", "dv", "dalpha", "dbeta_raw"):
            assert np.array_equal(res[key], whole[key][rows]), (n0, key)
        for key in ("S_T", "dS0"):
            assert np.array_equal(res[key], whole[key][n0:n1]), (n0, key)
        assert np.array_equal(res["saved"], whole["saved"][chunk_off[n0]:chunk_off[n1]])
        # every rank holds the same ordered sum of the partial gate gradients
        for key in ("da_log", "ddt_bias"):
            ref = whole[key]
            assert np.abs(res[key] - ref).max() <= 1e-12 * np.abs(ref).max(), key
            assert np.array_equal(res[key], parts[0][4][key])
    assert covered == inp.wl.total_tokens


def test_shard_ranges():
    sh = _sharding()
    assert sh.balanced_ranges(16, 3) == [(0, 6), (6, 11), (11, 16)]
    assert sh.balanced_ranges(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    h = sh.head_shard(16, 48, 4, 1)
    assert (h.kh0, h.kh1, h.h0, h.h1) == (4, 8, 12, 24)
    with pytest.raises(ValueError):
        sh.head_shard(16, 48, 2, 0, head_map=1)
    cu = [0, 100, 100, 350, 400, 1000]
    shards = [sh.sequence_shard(cu, 3, r) for r in range(3)]
    assert shards[0].n0 == 0 and shards[-1].n1 == 5
    for a, b in zip(shards, shards[1:]):
        assert a.n1 == b.n0 and a.t1 == b.t0
    assert sum(s.t1 - s.t0 for s in shards) == 1000
    for s in shards:
        assert s.cu_seqlens[0] == 0 and s.cu_seqlens[-1] == s.t1 - s.t0
