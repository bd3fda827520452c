"""Context parallelism: one long sequence cut into consecutive segments, one per worker.

The recurrence maps a segment's start state affinely to its end state.  Its token update
(lattice-inference 0.6.0, src/attention/gdn_backward.rs, module doc "Forward recap")
rewrites as S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T (k normalised), so

    S_out = Phi S_in + R,   Phi = prod_t g_t (I - beta_t k_t k_t^T)  (Dk x Dk, latest left),

with R the end state from a zero start.  Phi is itself the end state of the same
recurrence run with v = 0 from S_in = I (the value width then being Dk), so both come
from the forward kernels.  Reverse mode is affine the other way: the start-state gradient
is dS_in = Phi^T dS_out + G, G being dS_in when dS_out = 0.

Forward:  every segment forms (Phi, R) on its own; the pairs are all-gathered; each worker
          scans them, S_in(s) = Phi(s-1) S_in(s-1) + R(s-1) from S_in(0) = S_0, and runs
          its segment's forward from S_in(s).
Backward: every segment's backward with dS_out = 0 gives G(s); the G are all-gathered
          (the maps are kept from the forward's exchange, not sent again); each worker
          scans in reverse, dS_out(s) = Phi(s+1)^T dS_out(s+1) + G(s+1) from
          dS_out(last) = dS_T, and runs its segment's backward with dS_out(s).  d a_log and
          d dt_bias are sums over segments (an all-reduce); dS_0 is the first segment's.

The steps run through a backend (`GpuSegmentOps`: the library's C ABI) and a group
(`LocalGroup`: every segment in this process; `TorchGroup`: torch.distributed, the same
number of consecutive segments on every rank).  Cost per segment: two forwards to form
(Phi, R) and a third from the scanned start state; two backwards.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Any, List, Optional, Sequence


@dataclass
class Segment:
    """One segment's inputs (rows of the segment only) and the backend's per-segment
    state.  q, k, v, alpha, beta_raw: [L, *] rows; a_log, dt_bias: [Hv]."""
    q: Any
    k: Any
    v: Any
    alpha: Any
    beta_raw: Any
    a_log: Any
    dt_bias: Any
    state: dict = field(default_factory=dict)


class LocalGroup:
    """Every segment lives in this process: gathering is listing, reducing is adding."""

    def all_gather(self, local: List[Any]) -> List[Any]:
        return list(local)

    def all_reduce_sum(self, x):
        return x


class TorchGroup:
    """torch.distributed process group; every rank holds `per_rank` consecutive segments
    (rank r: global segments r*per_rank ... r*per_rank + per_rank - 1)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def all_gather(self, local: List[Any]) -> List[Any]:
        import torch
        stacked = torch.stack([t.contiguous() for t in local])
        parts = [torch.empty_like(stacked) for _ in range(self.dist.get_world_size(self.group))]
        self.dist.all_gather(parts, stacked, group=self.group)
        return [t for p in parts for t in p]

    def all_reduce_sum(self, x):
        self.dist.all_reduce(x, group=self.group)
        return x


@dataclass
class ForwardContext:
    """What forward() hands the backward() of the same segments: each local segment's
    start state and every segment's map, gathered once by the forward."""
    S_ins: List[Any]
    Phis: List[Any]
    n_local: int


def _first_index(group, n_local: int) -> int:
    if isinstance(group, TorchGroup):
        return group.dist.get_rank(group.group) * n_local
    return 0


def forward(ops, segments: Sequence[Segment], S0, group=None):
    """Returns ([o of each local segment], S_T of the whole sequence, a ForwardContext for
    the backward of the same segments).  S0: [1, Hv, Dk, Dv] start state or None (zero)."""
    group = group or LocalGroup()
    Phi_loc, R_loc = [], []
    for seg in segments:
        Phi_loc.append(ops.state_map(seg))
        R_loc.append(ops.forward(seg, None, keep=False)[1])
    Phis, Rs = group.all_gather(Phi_loc), group.all_gather(R_loc)
    first = _first_index(group, len(segments))
    S = ops.zero_state() if S0 is None else S0
    S_in_all = []
    for Phi, R in zip(Phis, Rs):
        S_in_all.append(S)
        S = ops.compose(Phi, S, R, transpose=False)
    outs, S_ins = [], []
    for j, seg in enumerate(segments):
        S_in = S_in_all[first + j]
        o, _ = ops.forward(seg, S_in, keep=True)
        outs.append(o)
        S_ins.append(S_in)
    return outs, S, ForwardContext(S_ins, list(Phis), len(segments))


def backward(ops, segments: Sequence[Segment], ctx: ForwardContext, dOs, dS_T, group=None):
    """Gradients of every local segment (dict per segment: dq, dk, dv, dalpha, dbeta_raw)
    and of the shared parameters summed over all segments (da_log, ddt_bias), plus dS_0
    (of the first segment; None on ranks that do not hold it).  `ctx` is what forward()
    returned for the same segments, run just before (the backend keeps its state)."""
    group = group or LocalGroup()
    if ctx.n_local != len(segments) or len(dOs) != len(segments):
        raise ValueError("backward: %d segments and %d dO for a forward of %d segments"
                         % (len(segments), len(dOs), ctx.n_local))
    S_ins, Phis = ctx.S_ins, ctx.Phis
    G_loc = [ops.backward(seg, S_in, dO, None)["dS0"]
             for seg, S_in, dO in zip(segments, S_ins, dOs)]
    Gs = group.all_gather(G_loc)
    if len(Phis) != len(Gs):
        raise ValueError("backward: %d gathered maps for %d segments" % (len(Phis), len(Gs)))
    first = _first_index(group, len(segments))
    n = len(Gs)
    dS_out = [None] * n
    d = ops.zero_state() if dS_T is None else dS_T
    for s in range(n - 1, -1, -1):
        dS_out[s] = d
        if s > 0:
            d = ops.compose(Phis[s], d, Gs[s], transpose=True)
    grads = []
    da_log = ddt = None
    for j, (seg, S_in, dO) in enumerate(zip(segments, S_ins, dOs)):
        g = ops.backward(seg, S_in, dO, dS_out[first + j])
        grads.append(g)
        da_log = g["da_log"] if da_log is None else da_log + g["da_log"]
        ddt = g["ddt_bias"] if ddt is None else ddt + g["ddt_bias"]
    da_log = group.all_reduce_sum(da_log)
    ddt = group.all_reduce_sum(ddt)
    dS0 = grads[0]["dS0"] if first == 0 else None
    return grads, da_log, ddt, dS0


class GpuSegmentOps:
    """The steps through the library's C ABI (all arithmetic in its kernels; PyTorch only
    allocates).  One sequence per segment."""

    def __init__(self, Hk, Hv, Dk, Dv, dtype, scale=0.0, device="cuda"):
        self.Hk, self.Hv, self.Dk, self.Dv = Hk, Hv, Dk, Dv
        self.dtype, self.scale, self.device = dtype, scale, device

    def _torch(self):
        import torch
        return torch

    def _layer(self, seg, key, Dv):
        import numpy as np
        import gated_deltanet_backward_gb300 as gdn
        if key not in seg.state:
            L = int(seg.q.shape[0])
            seg.state[key] = gdn.Layer.create(self.Hk, self.Hv, self.Dk, Dv,
                                              np.array([0, L], np.int32), self.dtype,
                                              self.scale, self.device)
        return seg.state[key]

    def zero_state(self):
        torch = self._torch()
        return torch.zeros(1, self.Hv, self.Dk, self.Dv, device=self.device)

    def state_map(self, seg):
        """Phi [1, Hv, Dk, Dk]: the end state of the recurrence with v = 0 from S_in = I."""
        torch = self._torch()
        L, Dk = int(seg.q.shape[0]), self.Dk
        layer = self._layer(seg, "map_layer", Dk)
        v0 = torch.zeros(L, self.Hv * Dk, device=self.device, dtype=seg.v.dtype)
        eye = torch.eye(Dk, device=self.device).expand(1, self.Hv, Dk, Dk).contiguous()
        o = torch.empty(L, self.Hv * Dk, device=self.device, dtype=seg.v.dtype)
        Phi = torch.empty(1, self.Hv, Dk, Dk, device=self.device)
        layer.forward(seg.q, seg.k, v0, seg.alpha, seg.beta_raw, seg.a_log, seg.dt_bias, eye, o,
                      Phi, keep_states=False)
        return Phi

    def forward(self, seg, S_in, keep):
        torch = self._torch()
        L = int(seg.q.shape[0])
        layer = self._layer(seg, "layer", self.Dv)
        o = torch.empty(L, self.Hv * self.Dv, device=self.device, dtype=seg.v.dtype)
        S_out = torch.empty(1, self.Hv, self.Dk, self.Dv, device=self.device)
        layer.forward(seg.q, seg.k, seg.v, seg.alpha, seg.beta_raw, seg.a_log, seg.dt_bias, S_in,
                      o, S_out, train=keep, keep_states=keep)
        return o, S_out

    def backward(self, seg, S_in, dO, dS_out):
        torch = self._torch()
        layer = seg.state["layer"]
        g = dict(dq=torch.empty_like(seg.q), dk=torch.empty_like(seg.k),
                 dv=torch.empty_like(seg.v), dalpha=torch.empty_like(seg.alpha),
                 dbeta_raw=torch.empty_like(seg.beta_raw), da_log=torch.empty_like(seg.a_log),
                 ddt_bias=torch.empty_like(seg.dt_bias),
                 dS0=torch.empty(1, self.Hv, self.Dk, self.Dv, device=self.device))
        layer.backward(seg.q, seg.k, seg.v, seg.alpha, seg.beta_raw, seg.a_log, seg.dt_bias, S_in,
                       dO, dS_out, g["dq"], g["dk"], g["dv"], g["dalpha"], g["dbeta_raw"],
                       g["da_log"], g["ddt_bias"], g["dS0"], train=True)
        return g

    def compose(self, Phi, S, R, transpose):
        """Phi S + R per head (Phi^T S + R with transpose), in the library's kernel."""
        import gated_deltanet_backward_gb300 as gdn
        out = self._torch().empty_like(R)
        gdn.gdn_state_compose(Phi, S, R, out, transpose)
        return out
