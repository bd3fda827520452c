"""Python binding of libgdn.so, the GB300 Gated DeltaNet library.

Argument marshalling only: every step of the forward and backward runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  The names
mirror the C ABI in ``include/gdn.h``:

    gdn_plan, gdn_saved_state_bytes, gdn_workspace_bytes,
    gdn_forward, gdn_backward, gdn_read_device_status, gdn_status_string

Tensors are passed as (data pointer, row stride); a 2-D tensor must have unit
column stride, so q/k/v may be column slices of one packed projection.  There
is no fallback: importing this package fails loudly when libgdn.so is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libgdn.so is not built (%s); run `python gated_deltanet_backward_gb300/build.py` "
        "or __graft_entry__.build()" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

GDN_OK = 0
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1
GDN_FLAG_KEEP_FOR_BACKWARD = 1
GDN_FLAG_REUSE_FORWARD = 2
GDN_FLAG_BF16_SAVED_STATES = 4
GDN_HEAD_MAP_CONSECUTIVE = 0
GDN_HEAD_MAP_MODULO = 1
GDN_ERR_NOT_KEPT = -8
CHUNK = 64


class gdn_shape(ctypes.Structure):
    _fields_ = [("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32),
                ("Dv", ctypes.c_int32), ("n_seqs", ctypes.c_int32),
                ("total_chunks", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("head_map", ctypes.c_int32)]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_SP = ctypes.POINTER(gdn_shape)
_I32P = ctypes.POINTER(ctypes.c_int32)

_lib.gdn_plan.argtypes = [_I32P, ctypes.c_int32, _I32P, _I32P]
_lib.gdn_plan.restype = ctypes.c_int
_lib.gdn_saved_state_bytes.argtypes = [_SP]
_lib.gdn_saved_state_bytes.restype = _sz
_lib.gdn_workspace_bytes.argtypes = [_SP, ctypes.c_int]
_lib.gdn_workspace_bytes.restype = _sz
# shape; q,k,v,alpha,beta_raw (+ld); a_log, dt_bias, cu, coff, S0; o (+ld); S_T, saved, ws,
# ws bytes, flags, stream
_u32 = ctypes.c_uint32
_lib.gdn_forward.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 5 + [_vp, _i64] +
                             [_vp, _vp, _vp, _sz, _u32, _vp])
_lib.gdn_forward.restype = ctypes.c_int
# as gdn_forward with z (+ld), gamma, eps, y (+ld) between saved_states and the workspace
_lib.gdn_forward_gated_rmsnorm.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 5 + [_vp, _i64] +
                                           [_vp, _vp] + [_vp, _i64, _vp, ctypes.c_float,
                                                         _vp, _i64] +
                                           [_vp, _sz, _u32, _vp])
_lib.gdn_forward_gated_rmsnorm.restype = ctypes.c_int
# shape; q,k,v,alpha,beta_raw (+ld); a_log, dt_bias, cu, coff, S0; dO (+ld); dS_T, saved;
# dq,dk,dv,dalpha,dbeta_raw (+ld); da_log, ddt_bias, dS0, ws, ws bytes, flags, stream
_lib.gdn_backward.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 5 + [_vp, _i64] + [_vp, _vp] +
                              [_vp, _i64] * 5 + [_vp, _vp, _vp, _vp, _sz, _u32, _vp])
_lib.gdn_backward.restype = ctypes.c_int
# as gdn_forward without the workspace, its size and the flags
_lib.gdn_forward_noalloc.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 5 + [_vp, _i64] +
                                     [_vp, _vp, _vp])
_lib.gdn_forward_noalloc.restype = ctypes.c_int
# shape; q,k,v,alpha,beta_raw (+ld); a_log, dt_bias, S_in, S_out; o (+ld); stream
_lib.gdn_decode_step.argtypes = [_SP] + [_vp, _i64] * 5 + [_vp] * 4 + [_vp, _i64, _vp]
_lib.gdn_decode_step.restype = ctypes.c_int
_lib.gdn_conv1d_silu_forward.argtypes = ([ctypes.c_int32, _i64, ctypes.c_int32, ctypes.c_int32,
                                          _vp, ctypes.c_int32, _vp, _i64, _vp, _vp, _i64, _vp])
_lib.gdn_conv1d_silu_forward.restype = ctypes.c_int
_lib.gdn_conv1d_silu_workspace_bytes.argtypes = [_i64, ctypes.c_int32, ctypes.c_int32]
_lib.gdn_conv1d_silu_workspace_bytes.restype = _sz
_lib.gdn_conv1d_silu_backward.argtypes = ([ctypes.c_int32, _i64, ctypes.c_int32, ctypes.c_int32,
                                           _vp, ctypes.c_int32, _vp, _i64, _vp, _vp, _i64, _vp,
                                           _i64, _vp, _vp, _sz, _vp])
_lib.gdn_conv1d_silu_backward.restype = ctypes.c_int
_lib.gdn_gated_rmsnorm_forward.argtypes = ([ctypes.c_int32, _i64, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_float] + [_vp, _i64] * 2 + [_vp, _vp, _i64,
                                                                                 _vp])
_lib.gdn_gated_rmsnorm_forward.restype = ctypes.c_int
_lib.gdn_gated_rmsnorm_workspace_bytes.argtypes = [ctypes.c_int32]
_lib.gdn_gated_rmsnorm_workspace_bytes.restype = _sz
_lib.gdn_gated_rmsnorm_backward.argtypes = ([ctypes.c_int32, _i64, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_float] + [_vp, _i64] * 2 + [_vp] +
                                            [_vp, _i64] * 3 + [_vp, _vp, _sz, _vp])
_lib.gdn_gated_rmsnorm_backward.restype = ctypes.c_int
_lib.gdn_state_compose.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp,
                                   _vp, ctypes.c_int32, _vp]
_lib.gdn_state_compose.restype = ctypes.c_int
_lib.gdn_kda_forward.argtypes = [_SP] + [_vp, _i64] * 5 + [_vp] * 5 + [_vp, _i64, _vp]
_lib.gdn_kda_forward.restype = ctypes.c_int
# shape; q,k,v,alpha,beta_raw (+ld); a_log, b_alpha, cu, coff, S_in, S_out; o (+ld); ws,
# ws bytes, stream
_lib.gdn_kda_forward_chunked.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 6 + [_vp, _i64] +
                                         [_vp, _sz, _vp])
_lib.gdn_kda_forward_chunked.restype = ctypes.c_int
_lib.gdn_kda_forward_chunked_workspace_bytes.argtypes = [_SP]
_lib.gdn_kda_forward_chunked_workspace_bytes.restype = _sz
_lib.gdn_kda_backward_workspace_bytes.argtypes = [_SP]
_lib.gdn_kda_backward_workspace_bytes.restype = _sz
_lib.gdn_kda_backward.argtypes = ([_SP] + [_vp, _i64] * 5 + [_vp] * 4 + [_vp, _i64] + [_vp] +
                                  [_vp, _i64] * 5 + [_vp] * 3 + [_vp, _sz, _vp])
_lib.gdn_kda_backward.restype = ctypes.c_int
_lib.gdn_read_device_status.argtypes = [_vp, _vp]
_lib.gdn_read_device_status.restype = ctypes.c_int
_lib.gdn_status_string.argtypes = [ctypes.c_int]
_lib.gdn_status_string.restype = ctypes.c_char_p
_lib.gdn_profile_begin.argtypes = [ctypes.POINTER(ctypes.c_void_p), _I32P, ctypes.c_int32]
_lib.gdn_profile_begin.restype = ctypes.c_int
_lib.gdn_profile_end.argtypes = []
_lib.gdn_profile_end.restype = ctypes.c_int
_lib.gdn_last_error.argtypes = []
_lib.gdn_last_error.restype = ctypes.c_char_p
_lib.gdn_kernel_name.argtypes = [ctypes.c_int32]
_lib.gdn_kernel_name.restype = ctypes.c_char_p

EXPORTED = ("gdn_plan", "gdn_saved_state_bytes", "gdn_workspace_bytes", "gdn_forward",
            "gdn_backward", "gdn_read_device_status", "gdn_status_string", "gdn_profile_begin",
            "gdn_profile_end", "gdn_kernel_name", "gdn_last_error", "gdn_forward_noalloc",
            "gdn_decode_step", "gdn_conv1d_silu_forward", "gdn_conv1d_silu_workspace_bytes",
            "gdn_conv1d_silu_backward", "gdn_gated_rmsnorm_forward",
            "gdn_gated_rmsnorm_workspace_bytes", "gdn_gated_rmsnorm_backward",
            "gdn_state_compose", "gdn_kda_forward", "gdn_kda_backward_workspace_bytes",
            "gdn_kda_backward", "gdn_forward_gated_rmsnorm", "gdn_kda_forward_chunked",
            "gdn_kda_forward_chunked_workspace_bytes")


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        if not detail and code == -4:
            detail = gdn_last_error()
        super().__init__("%s failed: %s (%d)%s" % (where, gdn_status_string(code), code,
                                                   (" -- " + detail) if detail else ""))


def gdn_last_error() -> str:
    return _lib.gdn_last_error().decode()


def gdn_status_string(code: int) -> str:
    return _lib.gdn_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != GDN_OK:
        raise GdnError(code, where)


def gdn_plan(cu_seqlens_host) -> tuple:
    """Host cu_seqlens -> (chunk_offsets int32 [n_seqs+1], total_chunks)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host), dtype=np.int32)
    n = len(cu) - 1
    off = np.zeros(n + 1, dtype=np.int32)
    tot = ctypes.c_int32(0)
    _check(_lib.gdn_plan(cu.ctypes.data_as(_I32P), n, off.ctypes.data_as(_I32P),
                         ctypes.byref(tot)), "gdn_plan")
    return off, int(tot.value)


def make_shape(Hk, Hv, Dk, Dv, n_seqs, total_chunks, total_tokens, dtype, scale=0.0,
               head_map=0) -> gdn_shape:
    """head_map: GDN_HEAD_MAP_CONSECUTIVE (0, key head h // (Hv // Hk)) or
    GDN_HEAD_MAP_MODULO (1, key head h % Hk)."""
    if not isinstance(dtype, int):
        dtype = GDN_DTYPE_BF16 if str(dtype) in ("bf16", "torch.bfloat16") else GDN_DTYPE_F32
    return gdn_shape(int(Hk), int(Hv), int(Dk), int(Dv), int(n_seqs), int(total_chunks),
                     int(total_tokens), int(dtype), float(scale or 0.0), int(head_map))


def gdn_saved_state_bytes(shape: gdn_shape) -> int:
    return int(_lib.gdn_saved_state_bytes(ctypes.byref(shape)))


def gdn_workspace_bytes(shape: gdn_shape, is_backward: bool) -> int:
    return int(_lib.gdn_workspace_bytes(ctypes.byref(shape), 1 if is_backward else 0))


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _mat(t):
    """(pointer, row stride in elements) of a 2-D tensor with unit column stride."""
    if t is None:
        return None, 0
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor, got shape %s" % (tuple(t.shape),))
    if t.numel() == 0:
        return int(t.data_ptr()), max(int(t.stride(0)), int(t.shape[1]))
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("columns must be contiguous (stride(1) == 1)")
    return int(t.data_ptr()), int(t.stride(0))


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _nbytes(t) -> int:
    return 0 if t is None else int(t.numel() * t.element_size())


F32, BF16, I32 = "torch.float32", "torch.bfloat16", "torch.int32"
_TOKEN_DTYPE = {GDN_DTYPE_F32: F32, GDN_DTYPE_BF16: BF16}
_TORCH = {}     # dtype name -> torch dtype, and whether CUDA is present (filled on first use)


def _torch_state():
    if not _TORCH:
        import torch
        _TORCH.update({F32: torch.float32, BF16: torch.bfloat16, I32: torch.int32,
                       "cuda": torch.cuda.is_available(), "torch": torch})
    return _TORCH


class _Call:
    """The tensors of one call, checked before any pointer reaches the library against
    what the call will read and write: the dtype, at least the rows and columns (or the
    elements, or the bytes) it touches, and then, after every size, that each tensor
    lives on the current CUDA device.  The library sees only pointers and strides, so a
    tensor that is too small, of another dtype or in host memory would otherwise be read
    or written out of its bounds.  A failed check raises GdnError with
    GDN_ERR_INVALID_ARG (GDN_ERR_UNSUPPORTED for an input dtype the library lacks) and
    calls nothing; a None is left to the library's own checks."""

    __slots__ = ("where", "tensors", "dt")

    def __init__(self, where: str):
        self.where = where
        self.tensors = []
        self.dt = _torch_state()

    def fail(self, detail: str, code: int = -1):
        raise GdnError(code, self.where, detail)

    def _dtype(self, t, name, dtype):
        if t.dtype is not self.dt[dtype]:
            self.fail("%s is %s, expected %s" % (name, t.dtype, dtype[len("torch."):]))

    def token_dtype(self, shape) -> str:
        if int(shape.dtype) not in _TOKEN_DTYPE:
            self.fail("shape.dtype %d is neither f32 nor bf16" % shape.dtype, -2)
        return _TOKEN_DTYPE[int(shape.dtype)]

    def io_dtype(self, t, name) -> str:
        if t is None or (t.dtype is not self.dt[F32] and t.dtype is not self.dt[BF16]):
            self.fail("%s must be a float32 or bfloat16 tensor" % name, -2)
        return F32 if t.dtype is self.dt[F32] else BF16

    def mat(self, t, name, rows, cols, dtype):
        """(pointer, row stride in elements) of a 2-D tensor of at least [rows, cols]
        with unit column stride; (None, 0) for None."""
        if t is None:
            return None, 0
        self.tensors.append((name, t))
        if t.dim() != 2:
            self.fail("%s must be 2-D, got shape %s" % (name, tuple(t.shape)))
        self._dtype(t, name, dtype)
        r, w = t.shape
        if r < rows or w < cols:
            self.fail("%s is %s, needs at least [%d, %d]" % (name, tuple(t.shape), rows, cols))
        s0, s1 = t.stride()
        if r == 0 or w == 0:
            return t.data_ptr(), max(s0, w)
        if w > 1 and s1 != 1:
            self.fail("%s needs contiguous columns (stride(1) == 1)" % name)
        return t.data_ptr(), s0

    def vec(self, t, name, numel, dtype):
        """Pointer of a contiguous tensor of at least `numel` elements, or None."""
        if t is None:
            return None
        self.tensors.append((name, t))
        self._dtype(t, name, dtype)
        if t.numel() < numel:
            self.fail("%s has %d elements, needs at least %d" % (name, t.numel(), numel))
        if not t.is_contiguous():
            self.fail("%s must be contiguous" % name)
        return t.data_ptr()

    def buf(self, t, name, nbytes=0):
        """Pointer of a contiguous buffer of at least `nbytes` bytes, or None."""
        if t is None:
            return None
        self.tensors.append((name, t))
        if _nbytes(t) < nbytes:
            self.fail("%s has %d bytes, needs at least %d" % (name, _nbytes(t), nbytes))
        if not t.is_contiguous():
            self.fail("%s must be contiguous" % name)
        return t.data_ptr()

    def ready(self):
        """Every tensor of the call on the current CUDA device (checked after the sizes)."""
        if not self.tensors:
            return
        dev = self.dt["torch"].cuda.current_device() if self.dt["cuda"] else -2
        for name, t in self.tensors:
            if not t.is_cuda or t.get_device() != dev:
                self.fail("%s is on %s, not on the current CUDA device" % (name, t.device))


def _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, rows, gate_cols,
                       tok):
    """Arguments q, k, v, alpha, beta_raw (each with its row stride), a_log, dt_bias of
    the recurrence's entry points (gate_cols: Hv, or Hv * Dk for the per-channel gate)."""
    Hk, Hv, Dk, Dv = int(shape.Hk), int(shape.Hv), int(shape.Dk), int(shape.Dv)
    args = []
    args += c.mat(q, "q", rows, Hk * Dk, tok)
    args += c.mat(k, "k", rows, Hk * Dk, tok)
    args += c.mat(v, "v", rows, Hv * Dv, tok)
    args += c.mat(alpha, "alpha", rows, gate_cols, F32)
    args += c.mat(beta_raw, "beta_raw", rows, Hv, F32)
    args += [c.vec(a_log, "a_log", Hv, F32),
             c.vec(dt_bias, "dt_bias" if gate_cols == Hv else "b_alpha", gate_cols, F32)]
    return args


def _state_elems(shape) -> int:
    return max(0, int(shape.n_seqs)) * max(0, int(shape.Hv)) * max(0, int(shape.Dk)) * \
        max(0, int(shape.Dv))


def gdn_forward(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, chunk_offsets, S0,
                o, S_T, saved_states, workspace, stream=None, flags=0) -> None:
    """Calls gdn_forward.  All tensors are CUDA tensors (S0 / S_T may be None).
    flags: GDN_FLAG_KEEP_FOR_BACKWARD (workspace then of the backward's size) and / or
    GDN_FLAG_BF16_SAVED_STATES (saved states as bf16 tiles instead of fp32)."""
    c = _Call("gdn_forward")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, T,
                               int(shape.Hv), tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32),
             c.vec(chunk_offsets, "chunk_offsets", N + 1, I32), c.vec(S0, "S0", ns, F32)]
    args += c.mat(o, "o", T, int(shape.Hv) * int(shape.Dv), tok)
    args += [c.vec(S_T, "S_T", ns, F32),
             c.buf(saved_states, "saved_states", gdn_saved_state_bytes(shape)),
             c.buf(workspace, "workspace"), _nbytes(workspace), int(flags)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_forward(*args), "gdn_forward")


def gdn_forward_gated_rmsnorm(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens,
                              chunk_offsets, S0, o, S_T, saved_states, z, gamma, eps, y,
                              workspace, stream=None, flags=0) -> None:
    """Calls gdn_forward_gated_rmsnorm: gdn_forward, and y = the gated RMSNorm of o with z,
    gamma [Dv] and eps over each (token, value head) row (fused into the forward's output
    pass for bf16)."""
    c = _Call("gdn_forward_gated_rmsnorm")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    wv = int(shape.Hv) * int(shape.Dv)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, T,
                               int(shape.Hv), tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32),
             c.vec(chunk_offsets, "chunk_offsets", N + 1, I32), c.vec(S0, "S0", ns, F32)]
    args += c.mat(o, "o", T, wv, tok)
    args += [c.vec(S_T, "S_T", ns, F32),
             c.buf(saved_states, "saved_states", gdn_saved_state_bytes(shape))]
    args += c.mat(z, "z", T, wv, tok)
    args += [c.vec(gamma, "gamma", int(shape.Dv), F32), float(eps)]
    args += c.mat(y, "y", T, wv, tok)
    args += [c.buf(workspace, "workspace"), _nbytes(workspace), int(flags)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_forward_gated_rmsnorm(*args), "gdn_forward_gated_rmsnorm")


def gdn_backward(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, chunk_offsets, S0,
                 dO, dS_T, saved_states, dq, dk, dv, dalpha, dbeta_raw, da_log, ddt_bias, dS0,
                 workspace, stream=None, flags=0) -> None:
    """Calls gdn_backward.  All tensors are CUDA tensors (S0, dS_T, dS0 may be None).
    flags: GDN_FLAG_REUSE_FORWARD (workspace then the one a keeping forward used) and /
    or GDN_FLAG_BF16_SAVED_STATES (as given to the forward that wrote saved_states)."""
    c = _Call("gdn_backward")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    Hv, wk, wv = int(shape.Hv), int(shape.Hk) * int(shape.Dk), int(shape.Hv) * int(shape.Dv)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, T, Hv, tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32),
             c.vec(chunk_offsets, "chunk_offsets", N + 1, I32), c.vec(S0, "S0", ns, F32)]
    args += c.mat(dO, "dO", T, wv, tok)
    args += [c.vec(dS_T, "dS_T", ns, F32),
             c.buf(saved_states, "saved_states", gdn_saved_state_bytes(shape))]
    args += c.mat(dq, "dq", T, wk, tok)
    args += c.mat(dk, "dk", T, wk, tok)
    args += c.mat(dv, "dv", T, wv, tok)
    args += c.mat(dalpha, "dalpha", T, Hv, F32)
    args += c.mat(dbeta_raw, "dbeta_raw", T, Hv, F32)
    args += [c.vec(da_log, "da_log", Hv, F32), c.vec(ddt_bias, "ddt_bias", Hv, F32),
             c.vec(dS0, "dS0", ns, F32), c.buf(workspace, "workspace"), _nbytes(workspace),
             int(flags)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_backward(*args), "gdn_backward")


def gdn_forward_noalloc(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens,
                        chunk_offsets, S0, o, S_T, saved_states, stream=None) -> None:
    """Calls gdn_forward_noalloc: the forward using the library's built-in scratch array
    instead of a caller workspace, for callers that cannot allocate device memory."""
    c = _Call("gdn_forward_noalloc")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, T,
                               int(shape.Hv), tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32),
             c.vec(chunk_offsets, "chunk_offsets", N + 1, I32), c.vec(S0, "S0", ns, F32)]
    args += c.mat(o, "o", T, int(shape.Hv) * int(shape.Dv), tok)
    args += [c.vec(S_T, "S_T", ns, F32),
             c.buf(saved_states, "saved_states", gdn_saved_state_bytes(shape))]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_forward_noalloc(*args), "gdn_forward_noalloc")


def gdn_decode_step(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, S_in, S_out, o,
                    stream=None) -> None:
    """Calls gdn_decode_step: one new token per sequence (row n of q, k, v, alpha,
    beta_raw, o); the state goes from S_in (None = zero) to S_out (may be S_in)."""
    c = _Call("gdn_decode_step")
    tok = c.token_dtype(shape)
    N, ns = int(shape.n_seqs), _state_elems(shape)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, dt_bias, N,
                               int(shape.Hv), tok)
    args += [c.vec(S_in, "S_in", ns, F32), c.vec(S_out, "S_out", ns, F32)]
    args += c.mat(o, "o", N, int(shape.Hv) * int(shape.Dv), tok)
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_decode_step(*args), "gdn_decode_step")


def _dtype_code(t) -> int:
    """gdn_dtype of a tensor: 1 for bfloat16, 0 for float32 (others are passed as -1, which
    the library rejects)."""
    name = str(t.dtype)
    return 1 if name == "torch.bfloat16" else 0 if name == "torch.float32" else -1


def gdn_conv1d_silu_workspace_bytes(total_tokens: int, channels: int, kernel_size: int) -> int:
    return int(_lib.gdn_conv1d_silu_workspace_bytes(int(total_tokens), int(channels),
                                                    int(kernel_size)))


def _conv_weights(c, w):
    if w is None or w.dim() != 2:
        c.fail("w must be a 2-D [channels, kernel_size] tensor")
    return int(w.shape[0]), int(w.shape[1])


def gdn_conv1d_silu_forward(x, w, cu_seqlens, y, stream=None) -> None:
    """Calls gdn_conv1d_silu_forward: x, y [T, C] (row strides taken from the tensors),
    w [C, K] fp32, cu_seqlens int32 [n_seqs + 1] on the device."""
    c = _Call("gdn_conv1d_silu_forward")
    dt = c.io_dtype(x, "x")
    C, K = _conv_weights(c, w)
    T = int(x.shape[0]) if x.dim() else 0
    xp, xld = c.mat(x, "x", T, C, dt)
    wp = c.vec(w, "w", C * K, F32)
    cp = c.vec(cu_seqlens, "cu_seqlens", 1, I32)
    yp, yld = c.mat(y, "y", T, C, dt)
    c.ready()
    n = int(cu_seqlens.numel()) - 1 if cu_seqlens is not None else 0
    _check(_lib.gdn_conv1d_silu_forward(_dtype_code(x), T, C, K, cp, n, xp, xld, wp, yp, yld,
                                        _stream(stream)), "gdn_conv1d_silu_forward")


def gdn_conv1d_silu_backward(x, w, cu_seqlens, dy, dx, dw=None, workspace=None,
                             stream=None) -> None:
    """Calls gdn_conv1d_silu_backward; dw (fp32 [C, K]) needs a workspace of
    gdn_conv1d_silu_workspace_bytes(T, C, K) bytes."""
    c = _Call("gdn_conv1d_silu_backward")
    dt = c.io_dtype(x, "x")
    C, K = _conv_weights(c, w)
    T = int(x.shape[0]) if x.dim() else 0
    xp, xld = c.mat(x, "x", T, C, dt)
    wp = c.vec(w, "w", C * K, F32)
    cp = c.vec(cu_seqlens, "cu_seqlens", 1, I32)
    gp, gld = c.mat(dy, "dy", T, C, dt)
    dp, dld = c.mat(dx, "dx", T, C, dt)
    dwp = c.vec(dw, "dw", C * K, F32)
    wsp = c.buf(workspace, "workspace")
    c.ready()
    n = int(cu_seqlens.numel()) - 1 if cu_seqlens is not None else 0
    _check(_lib.gdn_conv1d_silu_backward(_dtype_code(x), T, C, K, cp, n, xp, xld, wp, gp, gld,
                                         dp, dld, dwp, wsp, _nbytes(workspace), _stream(stream)),
           "gdn_conv1d_silu_backward")


def gdn_gated_rmsnorm_workspace_bytes(head_dim: int) -> int:
    return int(_lib.gdn_gated_rmsnorm_workspace_bytes(int(head_dim)))


def _norm_dims(c, o, gamma):
    if gamma is None or gamma.numel() == 0:
        c.fail("gamma must hold head_dim > 0 elements")
    if o.dim() != 2:
        c.fail("o must be 2-D, got shape %s" % (tuple(o.shape),))
    D = int(gamma.numel())
    return int(o.shape[0]), int(o.shape[1]) // D, D


def gdn_gated_rmsnorm_forward(o, z, gamma, y, eps, stream=None) -> None:
    """Calls gdn_gated_rmsnorm_forward: o, z, y [T, H*D] with D = gamma.numel()."""
    c = _Call("gdn_gated_rmsnorm_forward")
    dt = c.io_dtype(o, "o")
    T, H, D = _norm_dims(c, o, gamma)
    op, old = c.mat(o, "o", T, H * D, dt)
    zp, zld = c.mat(z, "z", T, H * D, dt)
    gp = c.vec(gamma, "gamma", D, F32)
    yp, yld = c.mat(y, "y", T, H * D, dt)
    c.ready()
    _check(_lib.gdn_gated_rmsnorm_forward(_dtype_code(o), T, H, D, float(eps), op, old, zp, zld,
                                          gp, yp, yld, _stream(stream)),
           "gdn_gated_rmsnorm_forward")


def gdn_gated_rmsnorm_backward(o, z, gamma, dy, d_o, dz, eps, dgamma=None, workspace=None,
                               stream=None) -> None:
    """Calls gdn_gated_rmsnorm_backward; dgamma (fp32 [D]) needs a workspace of
    gdn_gated_rmsnorm_workspace_bytes(D) bytes."""
    c = _Call("gdn_gated_rmsnorm_backward")
    dt = c.io_dtype(o, "o")
    T, H, D = _norm_dims(c, o, gamma)
    args = [_dtype_code(o), T, H, D, float(eps)]
    args += c.mat(o, "o", T, H * D, dt)
    args += c.mat(z, "z", T, H * D, dt)
    args += [c.vec(gamma, "gamma", D, F32)]
    args += c.mat(dy, "dy", T, H * D, dt)
    args += c.mat(d_o, "d_o", T, H * D, dt)
    args += c.mat(dz, "dz", T, H * D, dt)
    args += [c.vec(dgamma, "dgamma", D, F32), c.buf(workspace, "workspace"),
             _nbytes(workspace)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_gated_rmsnorm_backward(*args), "gdn_gated_rmsnorm_backward")


def gdn_state_compose(Phi, S, R, out, transpose=False, stream=None) -> None:
    """Calls gdn_state_compose: out[b] = op(Phi[b]) S[b] + R[b] over the leading blocks
    (Phi [..., Dk, Dk], S / R / out [..., Dk, Dv], fp32, contiguous; R may be None)."""
    c = _Call("gdn_state_compose")
    if S is None or S.dim() < 2:
        c.fail("S must be a [..., Dk, Dv] tensor")
    Dk, Dv = int(S.shape[-2]), int(S.shape[-1])
    n = int(S.numel()) // (Dk * Dv) if S.numel() else 0
    args = [n, Dk, Dv, c.vec(Phi, "Phi", n * Dk * Dk, F32), c.vec(S, "S", n * Dk * Dv, F32),
            c.vec(R, "R", n * Dk * Dv, F32), c.vec(out, "out", n * Dk * Dv, F32),
            1 if transpose else 0]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_state_compose(*args), "gdn_state_compose")


def gdn_kda_forward(shape, q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S_in, S_out, o,
                    stream=None) -> None:
    """Calls gdn_kda_forward: the per-channel-gate variant in token form (alpha
    [T, Hv*Dk], b_alpha [Hv*Dk]); S_in None = zero, S_out may be S_in."""
    c = _Call("gdn_kda_forward")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, b_alpha, T,
                               int(shape.Hv) * int(shape.Dk), tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32), c.vec(S_in, "S_in", ns, F32),
             c.vec(S_out, "S_out", ns, F32)]
    args += c.mat(o, "o", T, int(shape.Hv) * int(shape.Dv), tok)
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_kda_forward(*args), "gdn_kda_forward")


def gdn_kda_forward_chunked_workspace_bytes(shape) -> int:
    return int(_lib.gdn_kda_forward_chunked_workspace_bytes(ctypes.byref(shape)))


def gdn_kda_forward_chunked(shape, q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens,
                            chunk_offsets, S_in, S_out, o, workspace, stream=None) -> None:
    """Calls gdn_kda_forward_chunked: gdn_kda_forward as a chunked prefill on the tensor
    cores (bf16, Dk and Dv in {64, 128}); shape.total_chunks and chunk_offsets from
    gdn_plan; workspace of gdn_kda_forward_chunked_workspace_bytes(shape) bytes."""
    c = _Call("gdn_kda_forward_chunked")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, b_alpha, T,
                               int(shape.Hv) * int(shape.Dk), tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32),
             c.vec(chunk_offsets, "chunk_offsets", N + 1, I32), c.vec(S_in, "S_in", ns, F32),
             c.vec(S_out, "S_out", ns, F32)]
    args += c.mat(o, "o", T, int(shape.Hv) * int(shape.Dv), tok)
    args += [c.buf(workspace, "workspace", gdn_kda_forward_chunked_workspace_bytes(shape)),
             _nbytes(workspace)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_kda_forward_chunked(*args), "gdn_kda_forward_chunked")


def gdn_kda_backward_workspace_bytes(shape) -> int:
    return int(_lib.gdn_kda_backward_workspace_bytes(ctypes.byref(shape)))


def gdn_kda_backward(shape, q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S0, dO, dS_T,
                     dq, dk, dv, dalpha, dbeta_raw, da_log, db_alpha, dS0, workspace,
                     stream=None) -> None:
    """Calls gdn_kda_backward (S0, dS_T, dS0 may be None); workspace of
    gdn_kda_backward_workspace_bytes(shape) bytes."""
    c = _Call("gdn_kda_backward")
    tok = c.token_dtype(shape)
    T, N, ns = int(shape.total_tokens), int(shape.n_seqs), _state_elems(shape)
    Hv, Dk = int(shape.Hv), int(shape.Dk)
    wk, wv = int(shape.Hk) * Dk, Hv * int(shape.Dv)
    args = [ctypes.byref(shape)]
    args += _recurrence_inputs(c, shape, q, k, v, alpha, beta_raw, a_log, b_alpha, T, Hv * Dk,
                               tok)
    args += [c.vec(cu_seqlens, "cu_seqlens", N + 1, I32), c.vec(S0, "S0", ns, F32)]
    args += c.mat(dO, "dO", T, wv, tok)
    args += [c.vec(dS_T, "dS_T", ns, F32)]
    args += c.mat(dq, "dq", T, wk, tok)
    args += c.mat(dk, "dk", T, wk, tok)
    args += c.mat(dv, "dv", T, wv, tok)
    args += c.mat(dalpha, "dalpha", T, Hv * Dk, F32)
    args += c.mat(dbeta_raw, "dbeta_raw", T, Hv, F32)
    args += [c.vec(da_log, "da_log", Hv, F32), c.vec(db_alpha, "db_alpha", Hv * Dk, F32),
             c.vec(dS0, "dS0", ns, F32), c.buf(workspace, "workspace"), _nbytes(workspace)]
    c.ready()
    args.append(_stream(stream))
    _check(_lib.gdn_kda_backward(*args), "gdn_kda_backward")


def gdn_read_device_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the status word of a workspace."""
    c = _Call("gdn_read_device_status")
    wp = c.buf(workspace, "workspace", 4)
    c.ready()
    return int(_lib.gdn_read_device_status(wp, _stream(stream)))


def gdn_kernel_name(kernel_id: int) -> str:
    return _lib.gdn_kernel_name(int(kernel_id)).decode()


class gdn_profile:
    """Context manager around gdn_profile_begin / gdn_profile_end: brackets each kernel
    the library launches from this thread with two torch.cuda.Event's (recorded by the
    library on the launch's stream).  After exit and a synchronize, ``launches()`` gives
    (kernel name, milliseconds) per launch and ``count`` the launches seen."""

    def __init__(self, max_launches: int):
        import torch
        self.n = int(max_launches)
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * self.n)]
        for e in self.events:   # torch creates the CUDA event on its first record
            e.record()
        torch.cuda.current_stream().synchronize()
        self._handles = (ctypes.c_void_p * (2 * self.n))(
            *[ctypes.c_void_p(e.cuda_event) for e in self.events])
        self._ids = np.zeros(max(1, self.n), dtype=np.int32)
        self.count = 0

    def __enter__(self):
        _check(_lib.gdn_profile_begin(self._handles, self._ids.ctypes.data_as(_I32P), self.n),
               "gdn_profile_begin")
        return self

    def __exit__(self, *exc):
        self.count = int(_lib.gdn_profile_end())
        return False

    def launches(self):
        m = min(self.count, self.n)
        return [(gdn_kernel_name(self._ids[i]),
                 self.events[2 * i].elapsed_time(self.events[2 * i + 1])) for i in range(m)]


@dataclass
class Layer:
    """Device buffers for one varlen batch: shape, plan, saved states, workspaces.

    A convenience holder for callers of gdn_forward / gdn_backward; it only
    allocates (through PyTorch) and forwards arguments.  ``train=True`` runs the
    pair as a training step: the forward keeps the backward's chunk operands in
    the backward workspace (GDN_FLAG_KEEP_FOR_BACKWARD) and the backward reuses
    them (GDN_FLAG_REUSE_FORWARD) instead of recomputing them.
    """
    shape: gdn_shape
    cu_seqlens: object
    chunk_offsets: object
    saved_states: object
    ws_fwd: object
    ws_bwd: object
    bf16_states: bool = False   # GDN_FLAG_BF16_SAVED_STATES on both calls

    @classmethod
    def create(cls, Hk, Hv, Dk, Dv, cu_seqlens_host, dtype, scale=0.0, device="cuda",
               head_map=0, bf16_states=False):
        import torch
        off, nc = gdn_plan(cu_seqlens_host)
        cu = np.asarray(cu_seqlens_host, dtype=np.int32)
        shape = make_shape(Hk, Hv, Dk, Dv, len(cu) - 1, nc, int(cu[-1]), dtype, scale,
                           head_map)
        saved = torch.empty(max(4, gdn_saved_state_bytes(shape) // 4), dtype=torch.float32,
                            device=device)
        ws_f = torch.empty(max(256, gdn_workspace_bytes(shape, False)), dtype=torch.uint8,
                           device=device)
        ws_b = torch.empty(max(256, gdn_workspace_bytes(shape, True)), dtype=torch.uint8,
                           device=device)
        return cls(shape, torch.from_numpy(cu).to(device), torch.from_numpy(off).to(device),
                   saved, ws_f, ws_b, bool(bf16_states))

    def forward(self, q, k, v, alpha, beta_raw, a_log, dt_bias, S0, o, S_T, stream=None,
                train=False, keep_states=True):
        """keep_states=False (only without train) stores no chunk-start states: a
        forward that no backward reads (prefill, inference)."""
        gdn_forward(self.shape, q, k, v, alpha, beta_raw, a_log, dt_bias, self.cu_seqlens,
                    self.chunk_offsets, S0, o, S_T,
                    self.saved_states if (keep_states or train) else None,
                    self.ws_bwd if train else self.ws_fwd, stream,
                    (GDN_FLAG_KEEP_FOR_BACKWARD if train else 0) |
                    (GDN_FLAG_BF16_SAVED_STATES if self.bf16_states else 0))

    def backward(self, q, k, v, alpha, beta_raw, a_log, dt_bias, S0, dO, dS_T, dq, dk, dv,
                 dalpha, dbeta_raw, da_log, ddt_bias, dS0, stream=None, train=False):
        gdn_backward(self.shape, q, k, v, alpha, beta_raw, a_log, dt_bias, self.cu_seqlens,
                     self.chunk_offsets, S0, dO, dS_T, self.saved_states, dq, dk, dv, dalpha,
                     dbeta_raw, da_log, ddt_bias, dS0, self.ws_bwd, stream,
                     (GDN_FLAG_REUSE_FORWARD if train else 0) |
                     (GDN_FLAG_BF16_SAVED_STATES if self.bf16_states else 0))


__all__ = list(EXPORTED) + ["gdn_profile", "gdn_shape", "make_shape", "Layer", "GdnError", "LIB_PATH", "CHUNK",
                            "GDN_DTYPE_F32", "GDN_DTYPE_BF16", "GDN_FLAG_KEEP_FOR_BACKWARD",
                            "GDN_FLAG_REUSE_FORWARD", "GDN_FLAG_BF16_SAVED_STATES", "GDN_ERR_NOT_KEPT",
                            "GDN_HEAD_MAP_CONSECUTIVE", "GDN_HEAD_MAP_MODULO"]
