"""Data-parallel sharding of one batch of the recurrence over ranks (one process per GPU).

The work of the layer falls into (sequence, key-head group) units that are independent in
the forward and the backward: a key head's q/k rows are read only by its v_repeat value
heads (Gated Delta Networks, the head sharing of the 27B layer in the llama.cpp PR page
"tests: delta-net backward at the shape the 27B emits"), and a sequence never reads
another's tokens.  Two partitions follow, each a set of pointer offsets and a sub-shape
handed to the unchanged library:

* key-head groups: rank r owns key heads [kh0, kh1) (a balanced contiguous split of Hk)
  and the value heads that read them, h in [kh0 r, kh1 r) with the consecutive head map;
  its q / k / v / o / dq / dk / dv are column slices of the batch's row-major tensors
  (the same row strides), its alpha / beta_raw / dalpha / dbeta_raw column slices of the
  [T, Hv] gate matrices, its a_log / dt_bias / da_log / ddt_bias sub-vectors.  Nothing is
  exchanged: the ranks' outputs are disjoint slices of the whole batch's.
* sequences: rank r owns a contiguous range of whole sequences (balanced by tokens); its
  tensors are row slices.  d a_log and d dt_bias are per-head sums over every token of
  every sequence, so each rank's partial sums (2 Hv fp32) are all-gathered and added in
  rank order, which keeps the result independent of timing (no reduction whose order the
  collective picks).

The fp32 states S_0 / S_T / dS_T / dS_0 are [N, Hv, Dk, Dv] per batch; under either
partition a rank holds its own [N_r, Hv_r, Dk, Dv] block (a contiguous row slice under the
sequence split; the caller keeps per-rank blocks under the head split, where the heads of
one sequence are not contiguous across sequences).

Only the consecutive head map (value head h reads key head h / v_repeat) splits into
contiguous value-head ranges; the modulo map is refused here.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import numpy as np


def balanced_ranges(n: int, world: int) -> List[tuple]:
    """[start, end) of each of `world` contiguous parts of range(n), sizes differing by at
    most one (the first n % world parts one longer)."""
    if world < 1:
        raise ValueError("world must be >= 1")
    base, extra = divmod(n, world)
    out, s = [], 0
    for r in range(world):
        e = s + base + (1 if r < extra else 0)
        out.append((s, e))
        s = e
    return out


@dataclass(frozen=True)
class HeadShard:
    """Rank `rank`'s key heads [kh0, kh1) and value heads [h0, h1) of an (Hk, Hv) layer."""
    rank: int
    kh0: int
    kh1: int
    h0: int
    h1: int

    @property
    def Hk(self) -> int:
        return self.kh1 - self.kh0

    @property
    def Hv(self) -> int:
        return self.h1 - self.h0


def head_shard(Hk: int, Hv: int, world: int, rank: int, head_map: int = 0) -> HeadShard:
    if head_map != 0:
        raise ValueError("key-head sharding needs the consecutive head map (h / v_repeat)")
    if Hk <= 0 or Hv % Hk != 0:
        raise ValueError("Hv must be a positive multiple of Hk")
    if world > Hk:
        raise ValueError("more ranks (%d) than key heads (%d)" % (world, Hk))
    r = Hv // Hk
    kh0, kh1 = balanced_ranges(Hk, world)[rank]
    return HeadShard(rank, kh0, kh1, kh0 * r, kh1 * r)


def shard_heads(sh: HeadShard, Dk: int, Dv: int, *, q=None, k=None, v=None, alpha=None,
                beta_raw=None, a_log=None, dt_bias=None, dO=None, o=None, dq=None, dk=None,
                dv=None, dalpha=None, dbeta_raw=None, da_log=None, ddt_bias=None) -> dict:
    """The rank's views of the batch's tensors (numpy arrays or torch tensors; None stays
    None): column slices of the token-row tensors and sub-vectors of the per-head ones.
    No element is copied."""
    cols_k = slice(sh.kh0 * Dk, sh.kh1 * Dk)
    cols_v = slice(sh.h0 * Dv, sh.h1 * Dv)
    heads = slice(sh.h0, sh.h1)
    out = {}
    for name, t, sl in (("q", q, cols_k), ("k", k, cols_k), ("dq", dq, cols_k),
                        ("dk", dk, cols_k), ("v", v, cols_v), ("o", o, cols_v),
                        ("dO", dO, cols_v), ("dv", dv, cols_v), ("alpha", alpha, heads),
                        ("beta_raw", beta_raw, heads), ("dalpha", dalpha, heads),
                        ("dbeta_raw", dbeta_raw, heads)):
        out[name] = None if t is None else t[:, sl]
    for name, t in (("a_log", a_log), ("dt_bias", dt_bias), ("da_log", da_log),
                    ("ddt_bias", ddt_bias)):
        out[name] = None if t is None else t[heads]
    return out


@dataclass(frozen=True)
class SequenceShard:
    """Rank `rank`'s sequences [n0, n1) and their tokens [t0, t1) of a varlen batch."""
    rank: int
    n0: int
    n1: int
    t0: int
    t1: int
    cu_seqlens: np.ndarray      # the rank's own cu_seqlens (starting at 0)


def sequence_shard(cu_seqlens: Sequence[int], world: int, rank: int) -> SequenceShard:
    """Contiguous ranges of whole sequences with about equal tokens: the ranks' ranges
    meet at the sequence boundaries nearest to r T / world (r = 1 .. world - 1)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N, T = len(cu) - 1, int(cu[-1])
    if N < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("bad cu_seqlens, world or rank")

    def boundary(r):
        if r <= 0:
            return 0
        if r >= world:
            return N
        # the first of the nearest boundaries: non-decreasing in r
        return int(np.argmin(np.abs(cu - (r * T) // world)))

    n0, n1 = boundary(rank), boundary(rank + 1)
    t0, t1 = int(cu[n0]), int(cu[n1])
    return SequenceShard(rank, n0, n1, t0, t1, (cu[n0:n1 + 1] - t0).astype(np.int32))


def shard_sequences(sh: SequenceShard, **tensors) -> dict:
    """Row slices of the token-row tensors (name ending in nothing special) and of the
    per-sequence states (names S0, S_T, dS_T, dS0: rows n0 .. n1); per-head vectors
    (a_log, dt_bias) pass whole.  No element is copied."""
    rows = slice(sh.t0, sh.t1)
    seqs = slice(sh.n0, sh.n1)
    out = {}
    for name, t in tensors.items():
        if t is None:
            out[name] = None
        elif name in ("S0", "S_T", "dS_T", "dS0"):
            out[name] = t[seqs]
        elif name in ("a_log", "dt_bias", "da_log", "ddt_bias"):
            out[name] = t
        else:
            out[name] = t[rows]
    return out


def ordered_sum(parts):
    """Sum of the ranks' partial vectors in rank order (the same order on every run)."""
    total = parts[0] * 1
    for p in parts[1:]:
        total = total + p
    return total


def reduce_gate_grads(da_log, ddt_bias, group=None):
    """d a_log and d dt_bias of a sequence-sharded backward: every rank's partial sums,
    all-gathered and added in rank order (torch.distributed; one collective of 2 Hv
    values per rank).  Returns the totals on every rank."""
    import torch
    import torch.distributed as dist
    both = torch.stack([da_log, ddt_bias])
    parts = [torch.empty_like(both) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, both, group=group)
    total = ordered_sum(parts)
    return total[0], total[1]
