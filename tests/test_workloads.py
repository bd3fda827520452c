"""The seeded input generator (workloads/) that feeds both the oracle and the CUDA path:
the named workloads have the stated shapes, draws are reproducible byte for byte, bf16
workloads hold only bf16-exact values (rounded to nearest even, checked against
PyTorch's own conversion), packed q/k/v are views of one projection, and the
distributions are the stated ones."""
import numpy as np
import pytest

import workloads as W


def test_named_workloads_have_the_stated_shapes():
    t = W.get("tiny_f32")
    assert (t.dtype, t.Hk, t.Hv, t.Dk, t.Dv, t.seqlens, t.packed) == \
        ("f32", 2, 2, 16, 16, (64,), False)
    s = W.get("shared_kh_f32")
    assert (s.dtype, s.Hk, s.Hv, s.Dk, s.seqlens, s.v_repeat) == ("f32", 4, 12, 64, (512, 512), 3)
    l = W.get("l27b_bf16")
    assert (l.dtype, l.Hk, l.Hv, l.Dk, l.Dv, l.seqlens, l.row_width, l.total_chunks) == \
        ("bf16", 16, 48, 128, 128, (4096,), 10240, 64)
    b = W.get("l27b_batch_bf16")
    assert (b.n_seqs, b.total_tokens, b.S0_std, b.dST_std) == (8, 65536, 0.1, 0.01)
    v = W.get("varlen_bf16")
    assert (v.Hk, v.Hv, v.n_seqs) == (16, 32, 16)
    assert all(256 <= L <= 16384 for L in v.seqlens) and len(set(v.seqlens)) > 8
    assert list(v.cu_seqlens()) == [0] + list(np.cumsum(v.seqlens))


def test_draws_are_reproducible_and_seeded():
    wl = W.custom(dtype="bf16", Hk=2, Hv=4, Dk=32, Dv=16, seqlens=(40, 0, 9), seed=5,
                  S0_std=0.3, dST_std=0.2, dt_bias_std=0.1)
    a, b = W.generate(wl), W.generate(wl)
    for f in ("qkv", "alpha", "beta_raw", "a_log", "dt_bias", "S0", "dO", "dS_T"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = W.generate(W.replace(wl, seed=6))
    assert not np.array_equal(a.qkv, c.qkv)
    ls1, ls2 = W.generate_layer_steps(wl), W.generate_layer_steps(wl)
    assert np.array_equal(ls1.x, ls2.x) and np.array_equal(ls1.w, ls2.w)
    assert not np.array_equal(ls1.x, a.qkv)            # its own stream, not the recurrence's
    g1, g2 = W.generate_kda_gates(wl), W.generate_kda_gates(wl)
    assert np.array_equal(g1[0], g2[0]) and np.array_equal(g1[1], g2[1])


def test_bf16_workloads_hold_bf16_exact_values():
    torch = pytest.importorskip("torch")
    wl = W.custom(dtype="bf16", Hk=2, Hv=4, Dk=32, Dv=32, seqlens=(33, 7), seed=2)
    inp = W.generate(wl)
    for a in (inp.qkv, inp.dO):
        assert (a.view(np.uint32) & 0xFFFF).max() == 0
    ls = W.generate_layer_steps(wl)
    for a in (ls.x, ls.dy_conv, ls.o, ls.z, ls.dy_norm):
        assert (a.view(np.uint32) & 0xFFFF).max() == 0
    # round_bf16 against PyTorch's conversion, ties and extremes included
    x = np.concatenate([np.random.default_rng(0).standard_normal(4096).astype(np.float32) * 1e3,
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8),
                                  3.3895314e38, 1e-40, 0.0, -0.0], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(W.round_bf16(x).view(np.uint32), want.view(np.uint32))


def test_packed_qkv_are_views_of_one_projection():
    wl = W.custom(dtype="f32", Hk=2, Hv=6, Dk=16, Dv=8, seqlens=(10,), packed=True)
    inp = W.generate(wl)
    assert inp.qkv.shape == (10, 2 * 2 * 16 + 6 * 8)
    for a in (inp.q, inp.k, inp.v):
        assert np.shares_memory(a, inp.qkv)
    assert np.array_equal(inp.k, inp.qkv[:, 32:64]) and np.array_equal(inp.v, inp.qkv[:, 64:])


def test_distributions():
    wl = W.custom(dtype="f32", Hk=4, Hv=8, Dk=64, Dv=64, seqlens=(512, 512), seed=3,
                  S0_std=0.1, dST_std=0.01, dt_bias_std=0.2)
    inp = W.generate(wl)
    for a in (inp.qkv, inp.alpha, inp.beta_raw, inp.dO):   # N(0, 1): within 5 sigma
        n = a.size
        assert abs(a.mean()) < 5 / np.sqrt(n) and abs(a.std() - 1.0) < 5 / np.sqrt(2 * n)
    n = inp.S0.size
    assert abs(inp.S0.std() / 0.1 - 1) < 5 / np.sqrt(2 * n)
    assert abs(inp.dS_T.std() / 0.01 - 1) < 5 / np.sqrt(2 * n)
    assert inp.a_log.min() >= -1.0 and inp.a_log.max() <= 1.0
    assert inp.dt_bias.shape == (8,) and inp.dt_bias.std() > 0
    zero = W.generate(W.custom(dtype="f32", seqlens=(5,)))
    assert zero.S0 is None and zero.dS_T is None and not zero.dt_bias.any()
    ls = W.generate_layer_steps(wl, K=3, w_range=0.05)
    assert ls.w.shape == (wl.row_width, 3) and np.abs(ls.w).max() <= 0.05
    assert ls.gamma.min() >= 0.9 and ls.gamma.max() <= 1.1
    alpha, b_alpha = W.generate_kda_gates(wl)
    assert alpha.shape == (1024, 8 * 64) and b_alpha.shape == (8 * 64,)
    assert abs(b_alpha.std() / 0.2 - 1) < 5 / np.sqrt(2 * b_alpha.size)
    short = W.generate_layer_steps(wl, token_limit=600)
    assert list(short.cu_seqlens) == [0, 512, 600] and short.x.shape[0] == 600
