"""Seeded synthetic workloads for the Gated DeltaNet recurrence.

This module only draws random numbers and lays them out; it holds none of the
recurrence's arithmetic.  Both the CPU oracle (``oracle/``) and the CUDA path
consume exactly the arrays produced here, so the two sides always see the same
bytes (one draw threaded to both sides, as the KDA gradient work log on the
"dormouse" page recommends after its own reference drew a second input).

Shapes and distributions follow the five workloads of the layer:

* ``tiny_f32``      -- 1 x 64 tokens, Hk = Hv = 2, Dk = Dv = 16, dense q/k/v, fp32.
* ``shared_kh_f32`` -- 2 x 512 tokens, Hk = 4, Hv = 12, D = 64, packed strided qkv, fp32.
* ``l27b_bf16``     -- 1 x 4096 tokens, Hk = 16, Hv = 48, D = 128, packed qkv, bf16
                       (the 27B-shaped layer of the llama.cpp PR page: 16 key heads
                       shared by 48 value heads).
* ``l27b_batch_bf16`` -- 8 x 8192 tokens, same layer, bf16, nonzero S_0 and dS_T.
* ``varlen_bf16``   -- 16 sequences of U{256..16384} tokens, Hk = 16, Hv = 32, bf16.

``N(0, s)`` means standard deviation ``s``.  Draws use numpy's PCG64 generator
seeded with the workload's seed; the order of draws is fixed below.  bf16
workloads round every float draw to bf16 (round to nearest even) before either
side sees it, so the oracle upcasts exactly the values the GPU reads.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

CHUNK = 64  # tokens per chunk of the chunked GPU path (used only for sizes here)


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                  # "f32" or "bf16": type of q, k, v, o, dO, dq, dk, dv
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    seqlens: tuple              # tokens per sequence
    packed: bool = True         # q/k/v as row views of one packed buffer
    seed: int = 0
    dt_bias_std: float = 0.0    # 0 -> dt_bias = 0
    S0_std: float = 0.0         # 0 -> no initial state (S_0 = 0)
    dST_std: float = 0.0        # 0 -> no final-state adjoint (dS_T = 0)
    scale: Optional[float] = None  # None -> 1/sqrt(Dk)
    head_map: int = 0           # key head of value head h: 0 -> h // (Hv // Hk), 1 -> h % Hk

    @property
    def n_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def v_repeat(self) -> int:
        return self.Hv // self.Hk

    @property
    def row_width(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    @property
    def total_chunks(self) -> int:
        return int(sum((L + CHUNK - 1) // CHUNK for L in self.seqlens))

    def scale_value(self) -> float:
        return float(self.scale) if self.scale is not None else 1.0 / float(np.sqrt(self.Dk))

    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.n_seqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(np.asarray(self.seqlens, dtype=np.int64))
        return cu


def _varlen_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", 2, 2, 16, 16, (64,), packed=False, seed=0),
    "shared_kh_f32": Workload("shared_kh_f32", "f32", 4, 12, 64, 64, (512, 512), seed=1,
                              S0_std=0.1),
    "l27b_bf16": Workload("l27b_bf16", "bf16", 16, 48, 128, 128, (4096,), seed=2,
                          dt_bias_std=0.1),
    "l27b_batch_bf16": Workload("l27b_batch_bf16", "bf16", 16, 48, 128, 128, (8192,) * 8,
                                seed=3, S0_std=0.1, dST_std=0.01),
    "varlen_bf16": Workload("varlen_bf16", "bf16", 16, 32, 128, 128,
                            _varlen_lengths(4, 16, 256, 16384), seed=4,
                            S0_std=0.1, dST_std=0.01),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit fields (tests use this for edge cases)."""
    base = dict(dtype="f32", Hk=1, Hv=1, Dk=16, Dv=16, seqlens=(64,), packed=True, seed=0)
    base.update(kw)
    base["seqlens"] = tuple(int(x) for x in base["seqlens"])
    return Workload(name=name, **base)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    rounding = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((bits + rounding) & np.uint32(0xFFFF0000)).astype(np.uint32)
    return out.view(np.float32)


@dataclass
class Inputs:
    """One seeded draw.  Float arrays are float32 holding values exact in ``dtype``."""
    wl: Workload
    cu_seqlens: np.ndarray           # [N+1] int32
    qkv: Optional[np.ndarray]        # [T, 2*Hk*Dk + Hv*Dv] when packed
    q: np.ndarray                    # [T, Hk*Dk] (view of qkv when packed)
    k: np.ndarray                    # [T, Hk*Dk]
    v: np.ndarray                    # [T, Hv*Dv]
    alpha: np.ndarray                # [T, Hv] fp32
    beta_raw: np.ndarray             # [T, Hv] fp32
    a_log: np.ndarray                # [Hv] fp32
    dt_bias: np.ndarray              # [Hv] fp32
    S0: Optional[np.ndarray]         # [N, Hv, Dk, Dv] fp32 or None
    dO: np.ndarray                   # [T, Hv*Dv]
    dS_T: Optional[np.ndarray]       # [N, Hv, Dk, Dv] fp32 or None
    extra: dict = field(default_factory=dict)


def _normal(rng, shape, std=1.0):
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def generate(wl: Workload, token_limit: Optional[int] = None) -> Inputs:
    """Draw the inputs of ``wl``.  Draw order: qkv (or q, k, v), alpha, beta_raw,
    a_log, dt_bias, S_0, dO, dS_T."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    T = wl.total_tokens
    Hk, Hv, Dk, Dv = wl.Hk, wl.Hv, wl.Dk, wl.Dv
    cast = round_bf16 if wl.dtype == "bf16" else (lambda a: a)
    if wl.packed:
        qkv = cast(_normal(rng, (T, wl.row_width)))
        q = qkv[:, : Hk * Dk]
        k = qkv[:, Hk * Dk: 2 * Hk * Dk]
        v = qkv[:, 2 * Hk * Dk:]
    else:
        qkv = None
        q = cast(_normal(rng, (T, Hk * Dk)))
        k = cast(_normal(rng, (T, Hk * Dk)))
        v = cast(_normal(rng, (T, Hv * Dv)))
    alpha = _normal(rng, (T, Hv))
    beta_raw = _normal(rng, (T, Hv))
    a_log = rng.uniform(-1.0, 1.0, size=(Hv,)).astype(np.float32)
    dt_bias = (_normal(rng, (Hv,), wl.dt_bias_std) if wl.dt_bias_std > 0
               else np.zeros((Hv,), np.float32))
    S0 = _normal(rng, (wl.n_seqs, Hv, Dk, Dv), wl.S0_std) if wl.S0_std > 0 else None
    dO = cast(_normal(rng, (T, Hv * Dv)))
    dS_T = _normal(rng, (wl.n_seqs, Hv, Dk, Dv), wl.dST_std) if wl.dST_std > 0 else None
    return Inputs(wl, wl.cu_seqlens(), qkv, q, k, v, alpha, beta_raw, a_log, dt_bias,
                  S0, dO, dS_T)


__all__ = ["Workload", "Inputs", "WORKLOADS", "get", "custom", "generate", "round_bf16",
           "CHUNK", "replace"]


@dataclass
class LayerStepInputs:
    """One seeded draw for the layer steps either side of the recurrence.  Float arrays
    are float32 holding values exact in the workload's dtype (weights are fp32)."""
    cu_seqlens: np.ndarray           # [N+1] int32
    x: np.ndarray                    # [T, C] projection rows before the conv (q|k|v packed)
    w: np.ndarray                    # [C, K] conv weights, fp32
    dy_conv: np.ndarray              # [T, C] gradient of the conv output
    o: np.ndarray                    # [T, Hv*Dv] recurrence output
    z: np.ndarray                    # [T, Hv*Dv] gate projection
    gamma: np.ndarray                # [Dv] norm weight, fp32
    dy_norm: np.ndarray              # [T, Hv*Dv] gradient of the norm output


def generate_layer_steps(wl: Workload, K: int = 4, w_range: float = 0.05,
                         token_limit: Optional[int] = None) -> LayerStepInputs:
    """Inputs of the conv1d + SiLU and gated RMSNorm steps for ``wl``'s layer shape
    (C = 2 Hk Dk + Hv Dv channels, Hv heads of Dv).  Distributions follow the
    lattice-inference test model's initialisation: conv weights U(-w_range, w_range)
    (0.05 there), norm weights U(0.9, 1.1); the activations x, o, z and both incoming
    gradients are N(0, 1).  Seeded with seed + 7919 so it does not repeat the
    recurrence's draw.  Draw order: x, w, dy_conv, o, z, gamma, dy_norm."""
    rng = np.random.Generator(np.random.PCG64(wl.seed + 7919))
    T = wl.total_tokens if token_limit is None else min(wl.total_tokens, token_limit)
    lens, acc = [], 0
    for n in wl.seqlens:
        take = min(n, T - acc)
        if take <= 0 and acc >= T:
            break
        lens.append(take)
        acc += take
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    C = 2 * wl.Hk * wl.Dk + wl.Hv * wl.Dv
    W = wl.Hv * wl.Dv
    rnd = round_bf16 if wl.dtype == "bf16" else (lambda a: np.ascontiguousarray(a, np.float32))
    x = rnd(_normal(rng, (T, C)))
    w = rng.uniform(-w_range, w_range, size=(C, K)).astype(np.float32)
    dy_conv = rnd(_normal(rng, (T, C)))
    o = rnd(_normal(rng, (T, W)))
    z = rnd(_normal(rng, (T, W)))
    gamma = rng.uniform(0.9, 1.1, size=(wl.Dv,)).astype(np.float32)
    dy_norm = rnd(_normal(rng, (T, W)))
    return LayerStepInputs(cu, x, w, dy_conv, o, z, gamma, dy_norm)


def generate_kda_gates(wl: Workload, T: Optional[int] = None):
    """Per-channel decay-gate inputs of the KDA variant for ``wl``'s head shape: alpha
    [T, Hv*Dk] ~ N(0, 1) and b_alpha [Hv*Dk] ~ N(0, dt_bias_std) (zero when that is 0),
    fp32.  Seeded with seed + 104729; draw order alpha, b_alpha."""
    rng = np.random.Generator(np.random.PCG64(wl.seed + 104729))
    T = wl.total_tokens if T is None else T
    alpha = _normal(rng, (T, wl.Hv * wl.Dk))
    b_alpha = (_normal(rng, (wl.Hv * wl.Dk,), wl.dt_bias_std) if wl.dt_bias_std
               else np.zeros(wl.Hv * wl.Dk, np.float32))
    return alpha, b_alpha
