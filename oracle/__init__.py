"""CPU oracle for the Gated DeltaNet recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA product path never
touches it, and the two share no code: the only thing both sides consume is the
seeded draw of ``workloads``.

Contents
--------
* ``gdn_oracle.cpp`` -- token-by-token f64 forward and backward in C++
  (loaded here through ctypes; built by :func:`build`).
* ``chunked.py``     -- an f64 numpy restatement of the 64-token chunked (WY/UT)
  algebra that the GPU path uses, derived from the same recurrence.  It is
  pinned against the token-by-token oracle, never the other way round.
* ``chunked_kda.py`` -- the same chunked algebra for the KDA variant (a decay gate per
  key channel), with the Gram products formed by blocks of rows so that no factor
  overflows; pinned against the token-by-token KDA oracle.

Parity status: every function here is pinned by a ``-m "not gpu"`` test
(finite differences, closed forms, invariants, brute force); see
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with the host C++ compiler."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["g++"] + compile_flags() + [_SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


class _Shape(ctypes.Structure):
    _fields_ = [("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32),
                ("Dv", ctypes.c_int32), ("n_seqs", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("scale", ctypes.c_double),
                ("n_threads", ctypes.c_int32), ("segment", ctypes.c_int32),
                ("head_map", ctypes.c_int32)]


_P = ctypes.POINTER(ctypes.c_double)


class _Inputs(ctypes.Structure):
    _fields_ = [("q", _P), ("q_ld", ctypes.c_int64), ("k", _P), ("k_ld", ctypes.c_int64),
                ("v", _P), ("v_ld", ctypes.c_int64), ("alpha", _P), ("alpha_ld", ctypes.c_int64),
                ("beta_raw", _P), ("beta_ld", ctypes.c_int64), ("a_log", _P), ("dt_bias", _P),
                ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)), ("S0", _P)]


def open_library(path: str):
    """Load a build of ``gdn_oracle.cpp`` at ``path`` with the result types set.  The
    planted-mistake tests load edited builds this way and put them in place of the
    module's own library (``oracle._lib``) for the length of one test."""
    lib = ctypes.CDLL(path)
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_backward.restype = ctypes.c_int
    lib.gdn_oracle_forward_states.restype = ctypes.c_int
    lib.gdn_oracle_hardware_threads.restype = ctypes.c_int
    lib.gdn_oracle_state_map.restype = ctypes.c_int
    lib.gdn_oracle_kda_forward.restype = ctypes.c_int
    lib.gdn_oracle_kda_backward.restype = ctypes.c_int
    return lib


def compile_flags() -> list:
    """The host compiler flags every build of the oracle uses (strict IEEE f64: no fast
    math, no contraction into fused multiply-adds)."""
    return ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
            "-ffp-contract=off"]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def hardware_threads() -> int:
    return int(_load().gdn_oracle_hardware_threads())


def _f64(a) -> np.ndarray:
    """A C-contiguous-rows f64 array (row stride may exceed the width)."""
    a = np.asarray(a)
    if a.dtype != np.float64:
        a = a.astype(np.float64)
    if a.ndim == 2 and a.strides[1] == 8 and a.strides[0] % 8 == 0:
        return a
    return np.ascontiguousarray(a)


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.cast(None, _P)
    return a.ctypes.data_as(_P)


def _ld(a: np.ndarray) -> int:
    return a.strides[0] // 8


class _Args:
    """Holds f64 copies of one set of inputs alive while the C code runs."""

    def __init__(self, q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, S0, Hk, Hv, Dk, Dv,
                 scale, n_threads, segment, head_map=0):
        self.q, self.k, self.v = _f64(q), _f64(k), _f64(v)
        self.alpha, self.beta_raw = _f64(alpha), _f64(beta_raw)
        self.a_log = np.ascontiguousarray(a_log, dtype=np.float64)
        self.dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float64)
        self.cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        self.S0 = None if S0 is None else np.ascontiguousarray(S0, dtype=np.float64)
        self.T = int(self.cu[-1])
        self.N = int(len(self.cu) - 1)
        self.Hk, self.Hv, self.Dk, self.Dv = Hk, Hv, Dk, Dv
        self.shape = _Shape(Hk, Hv, Dk, Dv, self.N, self.T, float(scale or 0.0), int(n_threads),
                            int(segment), int(head_map))
        self.inputs = _Inputs(_ptr(self.q), _ld(self.q), _ptr(self.k), _ld(self.k), _ptr(self.v),
                              _ld(self.v), _ptr(self.alpha), _ld(self.alpha), _ptr(self.beta_raw),
                              _ld(self.beta_raw), _ptr(self.a_log), _ptr(self.dt_bias),
                              self.cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                              _ptr(self.S0))


def chunk_offsets(cu_seqlens, chunk: int) -> np.ndarray:
    """Chunk numbering: sequence n owns chunks [off[n], off[n+1])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = cu[1:] - cu[:-1]
    off = np.zeros(len(cu), dtype=np.int32)
    off[1:] = np.cumsum((lens + chunk - 1) // chunk)
    return off


def forward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, S0=None, *, Hk, Hv, Dk, Dv,
            scale=None, n_threads=0, chunk=0, head_map=0):
    """Token-by-token f64 forward.  Returns (o [T, Hv*Dv], S_T [N, Hv, Dk, Dv]), and when
    ``chunk`` > 0 also the state at the start of every chunk [NC, Hv, Dk, Dv].
    head_map 0: value head h reads key head h // (Hv // Hk); 1: key head h % Hk."""
    a = _Args(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, S0, Hk, Hv, Dk, Dv, scale,
              n_threads, 0, head_map)
    o = np.zeros((a.T, Hv * Dv), np.float64)
    S_T = np.zeros((a.N, Hv, Dk, Dv), np.float64)
    if chunk > 0:
        off = chunk_offsets(a.cu, chunk)
        states = np.zeros((int(off[-1]), Hv, Dk, Dv), np.float64)
        rc = _load().gdn_oracle_forward_states(
            ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(o), ctypes.c_int64(Hv * Dv),
            _ptr(S_T), ctypes.c_int32(chunk), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            _ptr(states))
    else:
        rc = _load().gdn_oracle_forward(ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(o),
                                        ctypes.c_int64(Hv * Dv), _ptr(S_T))
    if rc != 0:
        raise ValueError("gdn_oracle_forward rejected its arguments (%d)" % rc)
    return (o, S_T, states) if chunk > 0 else (o, S_T)


def backward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, dO, S0=None, dS_T=None, *,
             Hk, Hv, Dk, Dv, scale=None, n_threads=0, segment=64, head_map=0):
    """Token-by-token f64 backward.  Returns a dict of gradients:
    dq, dk [T, Hk*Dk] (summed over the value heads sharing a key head), dv [T, Hv*Dv],
    dalpha, dbeta_raw [T, Hv], da_log, ddt_bias [Hv], dS0 [N, Hv, Dk, Dv].
    head_map as for forward()."""
    a = _Args(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, S0, Hk, Hv, Dk, Dv, scale,
              n_threads, segment, head_map)
    dO = _f64(dO)
    dS_T = None if dS_T is None else np.ascontiguousarray(dS_T, dtype=np.float64)
    out = dict(dq=np.zeros((a.T, Hk * Dk)), dk=np.zeros((a.T, Hk * Dk)),
               dv=np.zeros((a.T, Hv * Dv)), dalpha=np.zeros((a.T, Hv)),
               dbeta_raw=np.zeros((a.T, Hv)), da_log=np.zeros(Hv), ddt_bias=np.zeros(Hv),
               dS0=np.zeros((a.N, Hv, Dk, Dv)))
    rc = _load().gdn_oracle_backward(
        ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(dO), ctypes.c_int64(_ld(dO)),
        _ptr(dS_T), _ptr(out["dq"]), ctypes.c_int64(Hk * Dk), _ptr(out["dk"]),
        ctypes.c_int64(Hk * Dk), _ptr(out["dv"]), ctypes.c_int64(Hv * Dv), _ptr(out["dalpha"]),
        ctypes.c_int64(Hv), _ptr(out["dbeta_raw"]), ctypes.c_int64(Hv), _ptr(out["da_log"]),
        _ptr(out["ddt_bias"]), _ptr(out["dS0"]))
    if rc != 0:
        raise ValueError("gdn_oracle_backward rejected its arguments (%d)" % rc)
    return out


def run_inputs(inp, which="both", n_threads=0, segment=64):
    """Run the oracle on a ``workloads.Inputs`` draw.  Returns (fwd, bwd) dicts."""
    wl = inp.wl
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, scale=wl.scale_value(), n_threads=n_threads,
              head_map=getattr(wl, "head_map", 0))
    fwd = bwd = None
    if which in ("both", "fwd"):
        o, S_T = forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                         inp.cu_seqlens, inp.S0, **kw)
        fwd = dict(o=o, S_T=S_T)
    if which in ("both", "bwd"):
        bwd = backward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias,
                       inp.cu_seqlens, inp.dO, inp.S0, inp.dS_T, segment=segment, **kw)
    return fwd, bwd


# ---------------------------------------------------------------------------
# The layer steps on either side of the recurrence (causal depthwise conv1d + SiLU
# before q/k/v, gated RMSNorm after o), f64.
def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def conv1d_silu_forward(x, w, cu_seqlens):
    """y[t, ch] = SiLU(sum_j w[ch, j] x[t - (K-1) + j, ch]), inputs before a sequence's start
    read as zero.  x [T, C], w [C, K]."""
    x = _f64(x)
    w = np.ascontiguousarray(w, dtype=np.float64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, C = x.shape
    y = np.zeros((T, C))
    rc = _load().gdn_oracle_conv1d_silu_forward(
        ctypes.c_int64(T), ctypes.c_int32(C), ctypes.c_int32(w.shape[1]),
        ctypes.c_int32(len(cu) - 1), _i32p(cu), _ptr(x), ctypes.c_int64(_ld(x)), _ptr(w),
        _ptr(y), ctypes.c_int64(C))
    if rc != 0:
        raise ValueError("gdn_oracle_conv1d_silu_forward rejected its arguments")
    return y


def conv1d_silu_backward(x, w, cu_seqlens, dy):
    """Returns (dx [T, C], dw [C, K])."""
    x, dy = _f64(x), _f64(dy)
    w = np.ascontiguousarray(w, dtype=np.float64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, C = x.shape
    dx = np.zeros((T, C))
    dw = np.zeros_like(w)
    rc = _load().gdn_oracle_conv1d_silu_backward(
        ctypes.c_int64(T), ctypes.c_int32(C), ctypes.c_int32(w.shape[1]),
        ctypes.c_int32(len(cu) - 1), _i32p(cu), _ptr(x), ctypes.c_int64(_ld(x)), _ptr(w),
        _ptr(dy), ctypes.c_int64(_ld(dy)), _ptr(dx), ctypes.c_int64(C), _ptr(dw))
    if rc != 0:
        raise ValueError("gdn_oracle_conv1d_silu_backward rejected its arguments")
    return dx, dw


def gated_rmsnorm_forward(o, z, gamma, H, D, eps):
    """y = (o / rms(o)) gamma SiLU(z) per (token, head); o, z [T, H*D], gamma [D]."""
    o, z = _f64(o), _f64(z)
    gamma = np.ascontiguousarray(gamma, dtype=np.float64)
    y = np.zeros((o.shape[0], H * D))
    rc = _load().gdn_oracle_gated_rmsnorm_forward(
        ctypes.c_int64(o.shape[0]), ctypes.c_int32(H), ctypes.c_int32(D), ctypes.c_double(eps),
        _ptr(o), ctypes.c_int64(_ld(o)), _ptr(z), ctypes.c_int64(_ld(z)), _ptr(gamma), _ptr(y),
        ctypes.c_int64(H * D))
    if rc != 0:
        raise ValueError("gdn_oracle_gated_rmsnorm_forward rejected its arguments")
    return y


def gated_rmsnorm_backward(o, z, gamma, dy, H, D, eps):
    """Returns (do, dz [T, H*D], dgamma [D])."""
    o, z, dy = _f64(o), _f64(z), _f64(dy)
    gamma = np.ascontiguousarray(gamma, dtype=np.float64)
    T = o.shape[0]
    d_o, dz, dg = np.zeros((T, H * D)), np.zeros((T, H * D)), np.zeros(D)
    rc = _load().gdn_oracle_gated_rmsnorm_backward(
        ctypes.c_int64(T), ctypes.c_int32(H), ctypes.c_int32(D), ctypes.c_double(eps), _ptr(o),
        ctypes.c_int64(_ld(o)), _ptr(z), ctypes.c_int64(_ld(z)), _ptr(gamma), _ptr(dy),
        ctypes.c_int64(_ld(dy)), _ptr(d_o), ctypes.c_int64(H * D), _ptr(dz),
        ctypes.c_int64(H * D), _ptr(dg))
    if rc != 0:
        raise ValueError("gdn_oracle_gated_rmsnorm_backward rejected its arguments")
    return d_o, dz, dg


# ---------------------------------------------------------------------------
# Context parallelism: the state map of a sequence, S_T = Phi S_0 + R.
def state_map(q, k, alpha, beta_raw, a_log, dt_bias, cu_seqlens, *, Hk, Hv, Dk, n_threads=0,
              head_map=0):
    """Phi [N, Hv, Dk, Dk] (f64): the product over a sequence's tokens of
    g_t (I - beta_t k_hat_t k_hat_t^T), latest token leftmost, so that the forward's final
    state is Phi S_0 + (the final state from S_0 = 0).  q is not read (any [T, Hk*Dk])."""
    T = int(np.asarray(cu_seqlens)[-1])
    v = np.zeros((T, Hv * Dk))
    a = _Args(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, None, Hk, Hv, Dk, Dk, None,
              n_threads, 0, head_map)
    Phi = np.zeros((a.N, Hv, Dk, Dk))
    rc = _load().gdn_oracle_state_map(ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(Phi))
    if rc != 0:
        raise ValueError("gdn_oracle_state_map rejected its arguments")
    return Phi


# ---------------------------------------------------------------------------
# KDA variant: a decay gate per key channel.  alpha [T, Hv*Dk], b_alpha [Hv*Dk]; channel c
# of value head h decays by exp(-exp(a_log[h]) softplus(alpha[t, h*Dk+c] + b_alpha[h*Dk+c])).
def kda_forward(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S0=None, *, Hk, Hv, Dk,
                Dv, scale=None, n_threads=0, head_map=0):
    """Token-by-token f64 KDA forward.  Returns (o [T, Hv*Dv], S_T [N, Hv, Dk, Dv])."""
    a = _Args(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S0, Hk, Hv, Dk, Dv, scale,
              n_threads, 0, head_map)
    o = np.zeros((a.T, Hv * Dv))
    S_T = np.zeros((a.N, Hv, Dk, Dv))
    rc = _load().gdn_oracle_kda_forward(ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(o),
                                        ctypes.c_int64(Hv * Dv), _ptr(S_T))
    if rc != 0:
        raise ValueError("gdn_oracle_kda_forward rejected its arguments")
    return o, S_T


def kda_backward(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, dO, S0=None, dS_T=None,
                 *, Hk, Hv, Dk, Dv, scale=None, n_threads=0, head_map=0):
    """Token-by-token f64 KDA backward (keeps every state: small shapes).  Returns dq, dk,
    dv, dalpha [T, Hv*Dk], dbeta_raw [T, Hv], da_log [Hv], db_alpha [Hv*Dk], dS0."""
    a = _Args(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S0, Hk, Hv, Dk, Dv, scale,
              n_threads, 0, head_map)
    dO = _f64(dO)
    dS_T = None if dS_T is None else np.ascontiguousarray(dS_T, dtype=np.float64)
    out = dict(dq=np.zeros((a.T, Hk * Dk)), dk=np.zeros((a.T, Hk * Dk)),
               dv=np.zeros((a.T, Hv * Dv)), dalpha=np.zeros((a.T, Hv * Dk)),
               dbeta_raw=np.zeros((a.T, Hv)), da_log=np.zeros(Hv), db_alpha=np.zeros(Hv * Dk),
               dS0=np.zeros((a.N, Hv, Dk, Dv)))
    rc = _load().gdn_oracle_kda_backward(
        ctypes.byref(a.shape), ctypes.byref(a.inputs), _ptr(dO), ctypes.c_int64(_ld(dO)),
        _ptr(dS_T), _ptr(out["dq"]), ctypes.c_int64(Hk * Dk), _ptr(out["dk"]),
        ctypes.c_int64(Hk * Dk), _ptr(out["dv"]), ctypes.c_int64(Hv * Dv), _ptr(out["dalpha"]),
        ctypes.c_int64(Hv * Dk), _ptr(out["dbeta_raw"]), ctypes.c_int64(Hv), _ptr(out["da_log"]),
        _ptr(out["db_alpha"]), _ptr(out["dS0"]))
    if rc != 0:
        raise ValueError("gdn_oracle_kda_backward rejected its arguments")
    return out
