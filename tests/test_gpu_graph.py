"""A training step (gdn_forward keeping its operands + gdn_backward reusing them) captured
into a CUDA graph: replays give the same bits as the uncaptured step.  The library's
launches (cooperative fused kernels, memsets) are stream-ordered and capturable, so a
caller can replay a fixed-shape step without per-launch host work."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


def test_captured_step_replays_bit_identically():
    torch = pytest.importorskip("torch")
    import gated_deltanet_backward_gb300 as gdn
    wl = W.custom(dtype="bf16", Hk=2, Hv=6, Dk=128, Dv=128, seqlens=(150, 70), seed=13,
                  S0_std=0.1, dST_std=0.01, dt_bias_std=0.1)
    inp = W.generate(wl)
    dev = lambda a, dt=torch.float32: (None if a is None else
                                       torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt))
    T, Hk, Hv, D, N = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.n_seqs
    bf = torch.bfloat16
    qkv = dev(inp.qkv, bf)
    q, k, v = qkv[:, :Hk * D], qkv[:, Hk * D:2 * Hk * D], qkv[:, 2 * Hk * D:]
    alpha, beta, a_log, dt_bias = (dev(x) for x in (inp.alpha, inp.beta_raw, inp.a_log,
                                                     inp.dt_bias))
    S0, dS_T, dO = dev(inp.S0), dev(inp.dS_T), dev(inp.dO, bf)
    layer = gdn.Layer.create(Hk, Hv, D, D, inp.cu_seqlens, "bf16", wl.scale_value())
    outs = dict(o=torch.empty(T, Hv * D, device="cuda", dtype=bf),
                S_T=torch.empty(N, Hv, D, D, device="cuda"),
                dq=torch.empty(T, Hk * D, device="cuda", dtype=bf),
                dk=torch.empty(T, Hk * D, device="cuda", dtype=bf),
                dv=torch.empty(T, Hv * D, device="cuda", dtype=bf),
                da=torch.empty(T, Hv, device="cuda"), db=torch.empty(T, Hv, device="cuda"),
                dal=torch.empty(Hv, device="cuda"), ddt=torch.empty(Hv, device="cuda"),
                dS0=torch.empty(N, Hv, D, D, device="cuda"))
    o = outs

    def step(st):
        layer.forward(q, k, v, alpha, beta, a_log, dt_bias, S0, o["o"], o["S_T"], st, train=True)
        layer.backward(q, k, v, alpha, beta, a_log, dt_bias, S0, dO, dS_T, o["dq"], o["dk"],
                       o["dv"], o["da"], o["db"], o["dal"], o["ddt"], o["dS0"], st, train=True)

    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        step(st)                      # first calls set kernel attributes outside the capture
    torch.cuda.synchronize()
    ref = {key: t.clone() for key, t in outs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        step(st)
    for _ in range(2):
        for t in outs.values():
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status(layer.ws_bwd) == 0
        for key, t in outs.items():
            assert torch.equal(t, ref[key]), key
