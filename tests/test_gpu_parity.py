"""GPU parity: the CUDA path (through the C ABI) against the f64 CPU oracle.

Bar per output tensor: max|gpu - oracle| / max|oracle| <= 1e-3 for fp32 inputs,
<= 2e-2 for bf16 inputs (an all-zero oracle tensor requires max|gpu| <= 1e-30).
Full-size workloads are checked on whole key-head groups (heads are independent,
so one group's oracle run covers every token of every sequence for those heads,
including the per-head sums d a_log / d dt_bias).
"""
import numpy as np
import pytest

import workloads as W
from tests.gdn_harness import (DeviceRun, TOL, compare, head_group_inputs, head_group_outputs,
                               oracle_outputs, rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _check_full(inp, dense=False):
    run = DeviceRun(inp, dense=dense)
    gpu = run.host()
    assert run.status() == 0 and run.status(backward=True) == 0
    ref = oracle_outputs(inp)
    return compare(gpu, ref, TOL[inp.wl.dtype]), run


def test_tiny_fp32_workload():
    """1 x 64 tokens, Hk = Hv = 2, D = 16, dense q/k/v, fp32."""
    _check_full(W.generate(W.get("tiny_f32")), dense=True)


def test_shared_key_heads_strided_fp32_workload():
    """2 x 512 tokens, 4 key heads shared by 12 value heads, packed strided qkv, fp32."""
    _check_full(W.generate(W.get("shared_kh_f32")))


@pytest.mark.parametrize("kw", [
    dict(Hk=1, Hv=2, Dk=16, Dv=16, seqlens=(200,)),                  # ragged 4th chunk
    dict(Hk=2, Hv=4, Dk=32, Dv=64, seqlens=(1, 65, 0, 130)),          # 1-token, empty, tails
    dict(Hk=1, Hv=3, Dk=128, Dv=32, seqlens=(70, 63)),                # Dk != Dv, large Dk
    dict(Hk=2, Hv=2, Dk=64, Dv=128, seqlens=(129,)),                  # Dv = 128, v_repeat 1
], ids=["T200_D16", "empty_and_1tok", "Dk128_Dv32", "Dk64_Dv128"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_shapes(kw, dtype):
    wl = W.custom(dtype=dtype, seed=7, S0_std=0.3, dST_std=0.2, dt_bias_std=0.2, **kw)
    _check_full(W.generate(wl))


def test_l27b_bf16_workload_full():
    """The 27B-shaped layer: 4096 tokens, Hk = 16, Hv = 48, D = 128, bf16 (every head)."""
    _check_full(W.generate(W.get("l27b_bf16")))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["l27b_batch_bf16", "varlen_bf16"])
def test_full_size_batches_on_every_head_group(name):
    """8 x 8192 tokens (Hv = 48) and the 16-sequence varlen batch (Hv = 32), run whole on
    the GPU; the oracle checks every key-head group (four at a time) over every token, so
    every output element of the batch is compared."""
    inp = W.generate(W.get(name))
    run = DeviceRun(inp)
    gpu = run.host()
    assert run.status() == 0 and run.status(backward=True) == 0
    del run
    Hk, step = inp.wl.Hk, 4
    worst = {}
    for kh in range(0, Hk, step):
        n = min(step, Hk - kh)
        sub = head_group_inputs(inp, kh, n)
        ref = oracle_outputs(sub)
        errs = compare(head_group_outputs(gpu, inp.wl, kh, n), ref, TOL["bf16"])
        for key, e in errs.items():
            worst[key] = max(worst.get(key, 0.0), e)
    print("worst max|err|/max|ref| over all key-head groups of %s: %s" % (name, worst))


def _bits(t):
    """A tensor's bytes as integers (so that NaN, -0 and +0 compare by their bits)."""
    import torch
    return t.view({torch.bfloat16: torch.int16, torch.float32: torch.int32}.get(t.dtype, t.dtype))


def _five_training_steps_are_byte_identical(inp):
    """Five complete training steps (forward keeping its operands, backward reusing them)
    on the same inputs: every output of every step equals the first step's byte for byte."""
    import torch
    run = DeviceRun(inp)
    assert run.status() == 0 and run.status(backward=True) == 0
    first = {k: v.clone() for k, v in run.device_outputs().items()}
    for step in range(4):
        run.run_forward()
        run.run_backward()
        assert run.status(backward=True) == 0
        for key, ref in first.items():
            assert torch.equal(_bits(run.device_outputs()[key]), _bits(ref)), (step, key)


def test_l27b_training_steps_are_byte_identical():
    """The 27B-shaped layer (the fused launches, with their work counters and flags)."""
    _five_training_steps_are_byte_identical(W.generate(W.get("l27b_bf16")))


@pytest.mark.slow
def test_l27b_batch_training_steps_are_byte_identical():
    """8 x 8192 tokens: more walks than SMs, so the separate launches run."""
    _five_training_steps_are_byte_identical(W.generate(W.get("l27b_batch_bf16")))


@pytest.mark.parametrize("name", ["small", "l27b_bf16"])
def test_bf16_saved_states_give_the_same_bits(name):
    """GDN_FLAG_BF16_SAVED_STATES keeps the chunk-start states as bf16 S^T tiles instead of
    fp32.  Every tensor-core product of the backward rounds the fp32 states to the same
    bf16 values, so o, S_T and every gradient are the same bits either way, and the tiles
    hold the fp32 states rounded to bf16."""
    import torch
    wl = W.get(name) if name != "small" else W.custom(
        dtype="bf16", Hk=2, Hv=6, Dk=128, Dv=64, seqlens=(300, 77), seed=41, S0_std=0.1,
        dST_std=0.05, dt_bias_std=0.1)
    inp = W.generate(wl)
    a = DeviceRun(inp)
    A = a.host()
    del a
    b = DeviceRun(inp, bf16_states=True)
    assert b.status() == 0 and b.status(backward=True) == 0
    B = b.host()
    del b
    for key in A:
        if key != "saved":
            assert np.array_equal(A[key], B[key]), key
    rounded = torch.from_numpy(A["saved"]).float().bfloat16().double().numpy()
    assert np.array_equal(B["saved"], rounded)


def test_strided_and_dense_inputs_give_identical_bits():
    inp = W.generate(W.custom(dtype="bf16", Hk=2, Hv=6, Dk=64, Dv=64, seqlens=(300, 77), seed=3,
                              S0_std=0.1, dST_std=0.1))
    a = DeviceRun(inp).host()
    b = DeviceRun(inp, dense=True).host()
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=False), key


def test_backward_is_bit_reproducible():
    import torch
    inp = W.generate(W.custom(dtype="bf16", Hk=4, Hv=12, Dk=64, Dv=64, seqlens=(256, 190),
                              seed=11, S0_std=0.1, dST_std=0.1))
    run = DeviceRun(inp)
    first = {k: v.clone() for k, v in run.grads.items()}
    for _ in range(4):
        again = run.run_backward()
        for key in first:
            assert torch.equal(again[key], first[key]), key


def test_zero_upstream_gives_zero_gradients():
    wl = W.custom(dtype="f32", Hk=2, Hv=4, Dk=32, Dv=32, seqlens=(100, 40), seed=5, S0_std=0.5)
    inp = W.generate(wl)
    inp.dO[:] = 0.0
    run = DeviceRun(inp)
    gpu = run.host()
    for key in ("dq", "dk", "dv", "dalpha", "dbeta_raw", "da_log", "ddt_bias", "dS0"):
        assert np.abs(gpu[key]).max() == 0.0, key


def test_all_empty_sequences():
    wl = W.custom(dtype="f32", Hk=1, Hv=2, Dk=16, Dv=16, seqlens=(0, 0), seed=2, S0_std=0.5,
                  dST_std=0.5)
    inp = W.generate(wl)
    gpu = DeviceRun(inp).host()
    assert np.array_equal(gpu["S_T"], inp.S0.astype(np.float64))
    assert np.array_equal(gpu["dS0"], inp.dS_T.astype(np.float64))
    assert np.abs(gpu["da_log"]).max() == 0.0 and np.abs(gpu["ddt_bias"]).max() == 0.0


def test_device_check_rejects_inconsistent_offsets():
    """chunk_offsets that disagree with cu_seqlens are caught by the kernels' own range
    checks (which run before any access) and reported through the status word."""
    import torch
    import gated_deltanet_backward_gb300 as gdn
    inp = W.generate(W.custom(dtype="f32", Hk=1, Hv=1, Dk=16, Dv=16, seqlens=(100, 100), seed=1))
    run = DeviceRun(inp, run_backward=False)
    assert run.status() == 0
    bad = torch.tensor([0, 1, 4], dtype=torch.int32, device="cuda")   # seq 0 has 2 chunks
    o = torch.zeros_like(run.o)
    gdn.gdn_forward(run.layer.shape, run.q, run.k, run.v, run.alpha, run.beta_raw, run.a_log,
                    run.dt_bias, run.layer.cu_seqlens, bad, None, o, None,
                    run.layer.saved_states, run.layer.ws_fwd)
    assert gdn.gdn_read_device_status(run.layer.ws_fwd) == -7


def test_saved_states_and_final_state_against_oracle_fp32():
    wl = W.custom(dtype="f32", Hk=2, Hv=4, Dk=32, Dv=16, seqlens=(150, 64, 3), seed=9,
                  S0_std=0.5)
    inp = W.generate(wl)
    gpu = DeviceRun(inp, run_backward=False).host()
    ref = oracle_outputs(inp, backward=False)
    assert rel_err(gpu["saved"], ref["saved"]) < 1e-4
    assert rel_err(gpu["S_T"], ref["S_T"]) < 1e-4


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_training_step_reuse_gives_the_bits_of_a_recomputing_backward(dtype):
    """A forward that keeps the chunk operands plus a backward that reuses them
    produce exactly the outputs of two calls that each compute everything."""
    wl = W.custom(dtype=dtype, Hk=2, Hv=6, Dk=128 if dtype == "bf16" else 32,
                  Dv=128 if dtype == "bf16" else 32, seqlens=(300, 0, 77, 64), seed=21,
                  S0_std=0.1, dST_std=0.1, dt_bias_std=0.1)
    inp = W.generate(wl)
    kept, fresh = DeviceRun(inp, train=True), DeviceRun(inp, train=False)
    assert kept.status() == 0 and kept.status(backward=True) == 0
    assert fresh.status() == 0 and fresh.status(backward=True) == 0
    a, b = kept.host(), fresh.host()
    for key in b:
        assert np.all(np.isfinite(a[key])), key
        assert np.array_equal(a[key], b[key]), key


def test_reuse_without_a_kept_forward_is_refused_on_the_device():
    """A reusing backward whose workspace holds no kept forward of its shape records
    GDN_ERR_NOT_KEPT and writes nothing; a proper training step afterwards works."""
    import gated_deltanet_backward_gb300 as gdn
    wl = W.custom(dtype="bf16", Hk=1, Hv=2, Dk=64, Dv=64, seqlens=(130, 40), seed=5)
    inp = W.generate(wl)
    # (1) the forward did not keep: its operands went to the forward workspace
    run = DeviceRun(inp, run_backward=False, train=False)
    run.layer.ws_bwd.zero_()
    g = run.run_backward(train=True)
    assert run.status(backward=True) == gdn.GDN_ERR_NOT_KEPT
    assert all(bool(t.isnan().all()) for t in g.values())
    # (2) the workspace was kept for another shape (a different output scale)
    run = DeviceRun(inp, run_backward=False, train=True)
    assert run.status() == 0
    run.layer.shape.scale = 0.5
    g = run.run_backward(train=True)
    assert run.status(backward=True) == gdn.GDN_ERR_NOT_KEPT
    assert all(bool(t.isnan().all()) for t in g.values())
    # (3) the context is intact: a training step on the same draw matches the oracle
    run = DeviceRun(inp, train=True)
    assert run.status() == 0 and run.status(backward=True) == 0
    compare(run.host(), oracle_outputs(inp), TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_without_saved_states_gives_the_same_bits(dtype):
    """A forward that keeps no chunk-start states (prefill / inference: saved_states =
    NULL) writes the same o and S_T, bit for bit, as one that keeps them, and leaves the
    saved-state buffer untouched."""
    import torch
    import gated_deltanet_backward_gb300 as gdn
    wl = W.custom(dtype=dtype, seed=11, Hk=2, Hv=4, Dk=64, Dv=64, seqlens=(130, 0, 70),
                  S0_std=0.3, dt_bias_std=0.2)
    run = DeviceRun(W.generate(wl), run_backward=False, train=False)
    o2 = torch.full_like(run.o, float("nan"))
    S_T2 = torch.full_like(run.S_T, float("nan"))
    run.layer.saved_states.fill_(7.0)
    run.layer.forward(run.q, run.k, run.v, run.alpha, run.beta_raw, run.a_log, run.dt_bias,
                      run.S0, o2, S_T2, keep_states=False)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(run.layer.ws_fwd) == 0
    assert torch.equal(o2.view(torch.int16 if dtype == "bf16" else torch.int32),
                       run.o.view(torch.int16 if dtype == "bf16" else torch.int32))
    assert torch.equal(S_T2.view(torch.int32), run.S_T.view(torch.int32))
    assert bool((run.layer.saved_states == 7.0).all())


@pytest.mark.parametrize("dtype,kw", [
    ("bf16", dict(Hk=2, Hv=6, Dk=64, Dv=64, seqlens=(130, 70))),
    ("f32", dict(Hk=2, Hv=6, Dk=32, Dv=64, seqlens=(100, 1))),
    ("bf16", dict(Hk=4, Hv=8, Dk=128, Dv=128, seqlens=(200,))),
], ids=["bf16_r3", "f32_r3", "bf16_r2_d128"])
def test_modulo_head_map_against_the_oracle(dtype, kw):
    """head_map = GDN_HEAD_MAP_MODULO (value head h reads key head h % Hk), forward and
    backward (training step and recomputing backward), against the oracle's modulo map."""
    wl = W.custom(dtype=dtype, seed=17, S0_std=0.3, dST_std=0.2, dt_bias_std=0.2, head_map=1,
                  **kw)
    inp = W.generate(wl)
    _, run = _check_full(inp)
    run.run_backward(train=False)
    compare(run.host(), oracle_outputs(inp), TOL[dtype],
            keys=["dq", "dk", "dv", "dalpha", "dbeta_raw", "da_log", "ddt_bias", "dS0"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_write_and_no_decay_leave_the_state_unchanged(dtype):
    """beta = 0 (beta_raw = -1000) and g = 1 (alpha = -1000: softplus = 0): nothing is
    written and nothing decays, so S_T is S_0 bit for bit and dv, d beta_raw are exactly
    zero; o and the rest of the gradients still match the oracle (o = scale S_0^T q_hat)."""
    wl = W.custom(dtype=dtype, Hk=2, Hv=4, Dk=64, Dv=64, seqlens=(100, 37), seed=29,
                  S0_std=0.5, dST_std=0.3, dt_bias_std=0.0)
    inp = W.generate(wl)
    inp.beta_raw[:] = -1000.0
    inp.alpha[:] = -1000.0
    gpu = DeviceRun(inp).host()
    assert np.array_equal(gpu["S_T"], inp.S0.astype(np.float64))
    assert np.abs(gpu["dv"]).max() == 0.0 and np.abs(gpu["dbeta_raw"]).max() == 0.0
    ref = oracle_outputs(inp)
    for key in ("o", "dq", "dS0"):
        assert rel_err(gpu[key], ref[key]) <= TOL[dtype], key
