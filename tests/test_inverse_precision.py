"""Design check for the chunk preparation's triangular inverse T = (I + A)^-1 (64 x 64,
A = diag(b) (E * K K^T) strictly lower; Gated Delta Networks, the WY / UT chunk form):
its 2x2 block merges, -D_1 A_10 D_0 at 32 x 32 and -T_B A_BA T_A at 64 x 64, are plain
matrix products that the tensor cores could form.  Every product that reads T reads it
as bf16 (the T diag(b) and T diag(b e^G) tiles), a relative step of 2^-9, so the merges
may add error well below that step and no more.  With the 16 x 16 diagonal inverses
exact and the merges fed rounded operands with fp32 accumulation:

* on chunks drawn like the 27B-layer and varlen workloads (their head shapes, key, gate
  and beta distributions), bf16 operands (kind::f16) and tf32 operands (kind::tf32)
  both stay under a quarter of the step;
* with nearly parallel keys and b near 1, where A's rows are largest (condition number
  ~70), tf32 operands stay under the step, while bf16 operands exceed it several times
  over: a tensor-core merge needs kind::tf32.

The reference is the f64 inverse.
"""
import numpy as np
import pytest

import workloads as W
from oracle import chunked

C = 64
BF16_STEP = 2.0 ** -9


def _round_bits(x, keep):
    """fp32 rounded to `keep` mantissa bits (nearest even), as fp32."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    drop = 23 - keep
    u = ((u + (1 << (drop - 1)) - 1 + ((u >> drop) & 1)) >> drop) << drop
    return u.astype(np.uint32).view(np.float32)


ROUND = {"bf16": lambda x: _round_bits(x, 7), "tf32": lambda x: _round_bits(x, 10)}


def _blocked_inverse(A, rnd):
    """The prep's doubling: 16 x 16 diagonal inverses (exact here), then the 32 x 32 and
    64 x 64 lower-left blocks as -D_1 (A_10 D_0), each product from rounded operands with
    fp32 accumulation (the intermediate rounded again as the second product's operand)."""
    f32 = lambda x: np.asarray(x, np.float32)
    A = f32(A)
    T = np.zeros_like(A)
    for b in range(0, C, 16):
        T[b:b + 16, b:b + 16] = f32(np.linalg.inv(np.eye(16) + A[b:b + 16, b:b + 16].astype(np.float64)))
    for q in (0, 32):
        D0, D1 = T[q:q + 16, q:q + 16], T[q + 16:q + 32, q + 16:q + 32]
        M = f32(rnd(A[q + 16:q + 32, q:q + 16]) @ rnd(D0))
        T[q + 16:q + 32, q:q + 16] = -f32(rnd(D1) @ rnd(M))
    M = f32(rnd(A[32:, :32]) @ rnd(T[:32, :32]))
    T[32:, :32] = -f32(rnd(T[32:, 32:]) @ rnd(M))
    return T


def _workload_chunks(name, n_chunks=6, n_heads=4):
    """A of the first chunks and value heads of a short draw shaped like a workload (its
    head shape, seed and gate distributions; 384 tokens)."""
    ref = W.get(name)
    wl = W.custom(dtype="bf16", seed=ref.seed, Hk=ref.Hk, Hv=ref.Hv, Dk=ref.Dk, Dv=ref.Dv,
                  seqlens=(C * n_chunks,), dt_bias_std=ref.dt_bias_std)
    inp = W.generate(wl)
    Dk, r = wl.Dk, wl.Hv // wl.Hk
    out = []
    for c in range(n_chunks):
        t = slice(C * c, C * (c + 1))
        for h in range(n_heads):
            K, _ = chunked._l2(inp.k[t, (h // r) * Dk:(h // r + 1) * Dk].astype(np.float64))
            x = inp.alpha[t, h].astype(np.float64) + inp.dt_bias[h]
            G = np.cumsum(-np.exp(inp.a_log[h]) * np.logaddexp(0.0, x))
            b = 1.0 / (1.0 + np.exp(-inp.beta_raw[t, h].astype(np.float64)))
            out.append(np.tril(b[:, None] * np.exp(G[:, None] - G[None, :]) * (K @ K.T), -1))
    return out


def _stress_chunks(n=6, seed=3):
    """Nearly parallel keys (a shared direction plus 5 % noise), b near 1, slow gates."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        base = rng.standard_normal(128)
        K, _ = chunked._l2(base[None, :] + 0.05 * rng.standard_normal((C, 128)))
        G = np.cumsum(-0.01 * rng.random(C))
        b = 0.95 + 0.05 * rng.random(C)
        out.append(np.tril(b[:, None] * np.exp(G[:, None] - G[None, :]) * (K @ K.T), -1))
    return out


def _worst(As, operands):
    worst = 0.0
    for A in As:
        T = np.linalg.inv(np.eye(C) + A)
        Tb = _blocked_inverse(A, ROUND[operands])
        assert np.isfinite(Tb).all()
        worst = max(worst, np.abs(Tb - T).max() / np.abs(T).max())
    return worst


@pytest.mark.parametrize("operands", ["bf16", "tf32"])
@pytest.mark.parametrize("source", ["l27b_bf16", "varlen_bf16"])
def test_merges_from_rounded_operands_on_workload_chunks(operands, source):
    worst = _worst(_workload_chunks(source), operands)
    assert worst < BF16_STEP / 4, worst      # measured: bf16 <= 3.7e-4, tf32 <= 3.4e-5


def test_merges_with_nearly_parallel_keys_need_tf32():
    As = _stress_chunks()
    tf32, bf16 = _worst(As, "tf32"), _worst(As, "bf16")
    assert tf32 < BF16_STEP, tf32            # measured ~1.4e-3
    assert bf16 > 2 * BF16_STEP, bf16        # measured ~1.1e-2
