"""Key-head sharding through the C ABI on one GPU: the shards of a batch (column views of
the same tensors, a sub-shape each) run one after another and give the unsharded run's
bits.  On a multi-GPU host each shard is one rank's work, with nothing exchanged."""
import importlib.util
import os
import sys

import numpy as np
import pytest

import workloads as W
from tests.gdn_harness import DeviceRun

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,world", [("bf16", 2), ("bf16", 3), ("f32", 2)])
def test_key_head_shards_give_the_unsharded_bits(dtype, world):
    import torch
    import gated_deltanet_backward_gb300 as gdn
    from gated_deltanet_backward_gb300 import sharding as shd
    wl = W.custom(dtype=dtype, Hk=6, Hv=18, Dk=64, Dv=64, seqlens=(300, 0, 130), seed=31,
                  S0_std=0.1, dST_std=0.05, dt_bias_std=0.1)
    inp = W.generate(wl)
    whole = DeviceRun(inp)
    ref = {k: v.clone() for k, v in whole.device_outputs().items()}
    T, N = wl.total_tokens, wl.n_seqs
    td = whole.tdtype
    outs = dict(o=torch.empty_like(whole.o), dq=torch.empty_like(whole.grads["dq"]),
                dk=torch.empty_like(whole.grads["dk"]), dv=torch.empty_like(whole.grads["dv"]),
                dalpha=torch.empty_like(whole.grads["dalpha"]),
                dbeta_raw=torch.empty_like(whole.grads["dbeta_raw"]),
                da_log=torch.empty_like(whole.grads["da_log"]),
                ddt_bias=torch.empty_like(whole.grads["ddt_bias"]))
    for rank in range(world):
        sh = shd.head_shard(wl.Hk, wl.Hv, world, rank)
        vw = shd.shard_heads(sh, wl.Dk, wl.Dv, q=whole.q, k=whole.k, v=whole.v,
                             alpha=whole.alpha, beta_raw=whole.beta_raw, a_log=whole.a_log,
                             dt_bias=whole.dt_bias, dO=whole.dO, **outs)
        hs = slice(sh.h0, sh.h1)
        S0 = whole.S0[:, hs].contiguous()          # the rank's own state blocks
        dS_T = whole.dS_T[:, hs].contiguous()
        S_T = torch.empty_like(S0)
        dS0 = torch.empty_like(S0)
        layer = gdn.Layer.create(sh.Hk, sh.Hv, wl.Dk, wl.Dv, inp.cu_seqlens, dtype,
                                 wl.scale_value())
        layer.forward(vw["q"], vw["k"], vw["v"], vw["alpha"], vw["beta_raw"], vw["a_log"],
                      vw["dt_bias"], S0, vw["o"], S_T, train=True)
        layer.backward(vw["q"], vw["k"], vw["v"], vw["alpha"], vw["beta_raw"], vw["a_log"],
                       vw["dt_bias"], S0, vw["dO"], dS_T, vw["dq"], vw["dk"], vw["dv"],
                       vw["dalpha"], vw["dbeta_raw"], vw["da_log"], vw["ddt_bias"], dS0,
                       train=True)
        assert gdn.gdn_read_device_status(layer.ws_bwd) == 0
        assert torch.equal(S_T, ref["S_T"][:, hs]), rank
        assert torch.equal(dS0, ref["dS0"][:, hs]), rank
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    for key, t in outs.items():
        assert torch.equal(bits(t), bits(ref[key])), key
