"""Throughput of the Gated DeltaNet forward + backward on GB300.

One step = gdn_forward followed by gdn_backward over one batch of the workload
(default: the 27B-shaped layer, 1 x 4096 tokens, 16 key heads shared by 48 value
heads, head size 128, bf16 q/k/v/o/dO, fp32 gates and state), inputs already
resident in HBM.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the launch stream, with an L2 flush between steps outside the events
(a 256 MB write, then a 256 MB read of another buffer: the 129 MB L2 then holds
none of the step's data and no dirty lines whose write-back the step would pay); barrier + synchronize around the timed loop;
max over ranks.  The library's profiling hook times every kernel launch of the
timed steps with CUDA events on the same stream, which gives the dominant
kernel's average duration for the roofline entry.

Multi-GPU: the work shards into independent (sequence, key-head group) units,
so N ranks each run their own batch with no data-path collective ("weak"
scaling); value = all ranks' tokens / the slowest rank's time.

--impl reference times the CPU oracle (f64, token by token, all host cores) on a
bounded sample of the same workload: the pages ship no runnable implementation.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "GDN fwd+bwd tokens/s (Hk16/Hv48, d128, bf16) and % of roofline on 1 GB300"
L2_FLUSH_BYTES = 256 << 20


def graph_step_times(fwd, bwd, flush, K, device, world):
    """The step (fwd(st), then bwd(st) if given: callables that launch on stream st)
    captured as CUDA graphs on a side stream and replayed K times there, each replay
    bracketed by CUDA events and the L2 flushed between steps.  Returns (step ms, forward
    ms, backward ms) averaged over the steps and maxed over the ranks, or None if the
    capture fails (the caller then reports the plain calls)."""
    import torch
    st = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    try:
        graphs = []
        for part in (fwd, bwd):
            if part is None:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                part(st)
            graphs.append(g)
    except Exception:
        torch.cuda.synchronize()
        return None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
          for _ in range(K)]
    with torch.cuda.stream(st):
        for _ in range(3):
            for g in graphs:
                g.replay()
            flush()
        for i in range(K):
            ev[i][0].record(st)
            for j, g in enumerate(graphs):
                g.replay()
                ev[i][j + 1].record(st)
            flush()
    torch.cuda.synchronize()
    parts = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) / K
             for j in range(len(graphs))]
    step = max_over_ranks(sum(parts), world, device)
    return step, parts[0], (parts[1] if len(parts) > 1 else 0.0)


class L2Flush:
    """Evicts the L2 between timed launches: writes one buffer larger than the L2, then
    reads another, so the writes' dirty lines are written back before the next timed
    launch instead of during it."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return dict(hbm_gbs=float(pk["hbm_gbs"]), bf16_tflops=float(pk["bf16_tflops"]),
                    bf16_tflops_sustained=float(pk.get("bf16_tflops_sustained",
                                                       pk["bf16_tflops"])),
                    sm_max_mhz=float(pk.get("sm_max_mhz", 2070.0)), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    sm_max_mhz=2070.0, source="fallback")


def alu_fp32_tflops(sm_mhz):
    """FP32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOP x clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------
# Algorithmic work model of the method (the headline roofline).  Per token it counts
# what the chunked method must move: the forward reads q, k, v, alpha, beta_raw and
# writes o and the fp32 chunk-start states (Hv Dk Dv 4 bytes per chunk); the backward
# reads q, k, v, alpha, beta_raw, dO and the states and writes dq, dk, dv, dalpha,
# dbeta_raw.  S_0 / S_T / dS_T / dS_0 add N Hv Dk Dv 4 bytes each where present.
# FLOPs are those of the chunked WY form (2 per multiply-add; triangular products at
# half), the Gram products shared by the v_repeat value heads of a key head, and the
# backward recomputing T, W, U and Delta.  The states count in fp32 whatever the
# library keeps, so the fraction does not depend on that choice.
# ----------------------------------------------------------------------------
def path_model(wl: W.Workload):
    es = 2 if wl.dtype == "bf16" else 4
    T, N, NC = wl.total_tokens, wl.n_seqs, wl.total_chunks
    Hk, Hv, Dk, Dv, C = wl.Hk, wl.Hv, wl.Dk, wl.Dv, W.CHUNK
    r = Hv // Hk
    qk = 2 * Hk * Dk * es
    v = Hv * Dv * es
    gates = 2 * Hv * 4
    states = NC * Hv * Dk * Dv * 4           # fp32 chunk-start states
    fwd = T * (qk + v + gates + v) + states
    bwd = T * (qk + v + gates + v) + states + T * (qk + v + gates)
    st = N * Hv * Dk * Dv * 4
    fwd += st * ((wl.S0_std > 0) + 1)
    bwd += st * ((wl.S0_std > 0) + (wl.dST_std > 0) + 1)
    # chunked-method FLOPs per chunk and value head; the Gram products K K^T and Q K^T
    # are formed once per key head and shared by its r value heads
    gram = 2 * C * C * Dk / r
    f_fwd = (2 * gram + C ** 3 / 3                    # K K^T, Q K^T; T = (I + A)^-1
             + 2 * C * C * Dk + 2 * C * C * Dv        # W, U
             + 2 * C * C * Dv + 6 * C * Dk * Dv)      # P Delta; W S, Q S, K^T Delta
    f_bwd = (2 * gram + C ** 3 / 3 + 2 * C * C * (Dk + Dv) + 2 * C * Dk * Dv   # recompute
             + 2 * C * C * Dv + 6 * C * Dk * Dv       # dDelta and the dS carry
             + 6 * C * C * Dv + 12 * C * C * Dk + 6 * C * Dk * Dv + 4 * C ** 3)  # chunk VJP
    return dict(bytes_fwd=fwd, bytes_bwd=bwd, bytes=fwd + bwd, flops_fwd=NC * Hv * f_fwd,
                flops_bwd=NC * Hv * f_bwd, flops=NC * Hv * (f_fwd + f_bwd),
                bytes_per_token=(fwd + bwd) / max(T, 1), flops_per_token=NC * Hv *
                (f_fwd + f_bwd) / max(T, 1))


# The kernels of each pass: a pass's algorithmic work (path_model) is what its kernels
# do between them; a fused pass is one launch.
FWD_KERNELS = ("gdn_fwd_fused_tc", "gdn_prep_tc", "gdn_prep_tc_full", "gdn_fwd_state_tc",
               "gdn_fwd_out_tc", "gdn_prep", "gdn_fwd_state")
BWD_KERNELS = ("gdn_bwd_fused_tc", "gdn_bwd_state_tc", "gdn_bwd_grads_tc", "gdn_bwd_state",
               "gdn_bwd_grads", "gdn_bwd_qk", "gdn_bwd_gates")


def kernel_models(wl: W.Workload):
    """kernel name -> (implementation bytes per launch, FLOPs per launch, compute unit).

    Implementation bytes: each kernel's compulsory reads and writes of its own inputs
    and outputs in this library's decomposition, workspace intermediates (the operand
    tiles one kernel hands the next) included.  A diagnostic beside the measured DRAM
    traffic, not the method's algorithmic work (path_model)."""
    es = 2 if wl.dtype == "bf16" else 4
    NC, N = wl.total_chunks, wl.n_seqs
    Hk, Hv, Dk, Dv, C = wl.Hk, wl.Hv, wl.Dk, wl.Dv, W.CHUNK
    r = Hv // Hk
    T = wl.total_tokens
    f4 = 4
    prep_b = (T * (2 * Hk * Dk * es + Hv * Dv * es + 2 * Hv * 4) +
              NC * Hk * C * (2 * Dk + 2) * f4 + NC * Hv * C * (Dk + Dv + 2) * f4)
    prep_f = NC * Hk * (2 * C * C * Dk + r * (C ** 3 / 3 + 2 * C * C * (Dk + Dv)))
    fst_b = (NC * Hk * C * 2 * Dk * f4 + NC * Hv * C * (Dk + Dv + 1) * f4 + T * Hv * Dv * es +
             NC * Hv * Dk * Dv * f4)
    fst_f = NC * Hv * (6 * C * Dk * Dv + C * C * Dv) + NC * Hk * 2 * C * C * Dk
    bst_b = (NC * Hk * C * 2 * Dk * f4 + NC * Hv * C * (Dk + 1) * f4 + T * Hv * Dv * es +
             NC * Hv * (Dk * Dv + C * Dv) * f4)
    bst_f = NC * Hv * (C * C * Dv + 6 * C * Dk * Dv) + NC * Hk * 2 * C * C * Dk
    bgr_b = (NC * Hv * (2 * Dk * Dv + C * (Dk + 2 * Dv + C + 3)) * f4 +
             NC * Hk * C * 2 * Dk * f4 + T * Hv * 2 * Dv * es + T * Hv * 4 +
             NC * Hv * 2 * C * Dk * f4 + T * Hv * Dv * es + T * Hv * 2 * 4)
    bgr_f = NC * Hv * (12 * C * Dk * Dv + 2 * C * C * (5 * Dk + 3 * Dv) + 4 * C ** 3)
    bqk_b = NC * Hv * 2 * C * Dk * f4 + NC * Hk * C * 2 * (Dk + 1) * f4 + T * Hk * 2 * Dk * es
    # tensor-core (bf16) kernels: every operand handed between kernels is a bf16
    # 128B-swizzled tile; the bytes below are each kernel's reads plus writes of
    # distinct data (a key-head tile read by its r value-head CTAs counts once)
    sKC = (Dk + 63) // 64 * C * 128                  # [C][Dk] tile
    sVC = (Dv + 63) // 64 * C * 128                  # [C][Dv] tile
    sVt, sCC = Dv * 128, C * C * 2                   # [Dv][C], [C][C] tiles
    MV = max(Dv, 64)
    sST = (Dk + 63) // 64 * MV * 128                 # S^T / dS^T state tile [MV][Dk]
    tok_in = T * (2 * Hk * Dk * es + Hv * Dv * es + 2 * Hv * 4)   # q, k, v, alpha, beta
    tc_prep_b = (tok_in + NC * Hk * 2 * sKC +                       # Q, K tiles
                 NC * Hv * (2 * C * 4 + sVt + sKC + sCC))           # G, b, U^T, W, P
    tc_prep_f = (NC * Hk * 2 * 128 * C * Dk + NC * Hv * (2 * C * C * (Dk + Dv) + C ** 3 / 3 +
                                                          C * C * 8))
    tc_prep_bwd_b = tc_prep_b + (NC * Hk * (2 * C * 4 + C * C * 4) +   # norms, K K^T
                                 NC * Hv * 2 * sCC)                   # T, T diag(b e^G)
    st = N * Hv * Dk * Dv * 4
    fst_st = st * ((wl.S0_std > 0) + 1)                             # S0 read, S_T written
    bst_st = st * ((wl.dST_std > 0) + 1)                            # dS_T read, dS0 written
    fst_tc_b = (NC * Hk * 2 * sKC + NC * Hv * (sKC + sCC + sVt + C * 4) +
                T * Hv * Dv * es + NC * Hv * sST + fst_st)          # ... o, saved S^T tiles
    fst_tc_f = NC * Hv * (6 * C * Dk * Dv + 2 * C * C * Dv)
    bst_tc_b = (NC * Hk * 2 * sKC + NC * Hv * (sCC + sKC + C * 4) + T * Hv * Dv * es +
                NC * Hv * (sST + sVC) + bst_st)                     # ... dS^T, -dDelta
    bst_tc_f = NC * Hv * (2 * C * C * Dv + 6 * C * Dk * Dv)
    bgr_tc_b = (NC * Hk * (2 * sKC + C * C * 4 + 2 * C * 4) + T * Hk * 2 * Dk * es +
                NC * Hv * (sST + 2 * C * 4 + sKC + sVt + 2 * sVC + sCC + sST + 2 * sCC + 8) +
                T * Hv * (2 * Dv * es + 4) + T * Hv * (Dv * es + 8))
    bgr_tc_f = NC * Hv * (2 * C * Dk * Dv + 2 * 128 * Dk * Dv + 2 * C * Dk * Dv +
                          4 * C * Dk * Dv + 2 * C * C * Dv + 2 * C * C * (Dv + Dk) +
                          4 * C * C * Dk + 2 * C * C * Dv + 4 * C ** 3 + 4 * C * C * Dk +
                          2 * C * C * Dk)
    # output pass: Q tiles, the walk's S^T and Delta^T tiles, P and G in, o out
    out_tc_b = (NC * Hk * sKC + NC * Hv * (sST + MV * 128 + sCC + C * 4) + T * Hv * Dv * es)
    out_tc_f = NC * Hv * (2 * C * Dk * Dv + 2 * C * C * Dv)
    return {
        "gdn_fwd_out_tc": (out_tc_b, out_tc_f, "tensor"),
        "gdn_fwd_fused_tc": (tc_prep_bwd_b + fst_tc_b, tc_prep_f + fst_tc_f, "tensor"),
        "gdn_bwd_fused_tc": (bst_tc_b + bgr_tc_b, bst_tc_f + bgr_tc_f, "tensor"),
        "gdn_prep_tc": (tc_prep_b, tc_prep_f, "tensor"),
        "gdn_prep_tc_full": (tc_prep_bwd_b, tc_prep_f, "tensor"),
        "gdn_fwd_state_tc": (fst_tc_b, fst_tc_f, "tensor"),
        "gdn_bwd_state_tc": (bst_tc_b, bst_tc_f, "tensor"),
        "gdn_bwd_grads_tc": (bgr_tc_b, bgr_tc_f, "tensor"),
        "gdn_prep": (prep_b, prep_f, "alu"),
        "gdn_fwd_state": (fst_b, fst_f, "alu"),
        "gdn_bwd_state": (bst_b, bst_f, "alu"),
        "gdn_bwd_grads": (bgr_b, bgr_f, "alu"),
        "gdn_bwd_qk": (bqk_b, 0.0, "alu"),
        "gdn_bwd_gates": (NC * Hv * 8 + Hv * 8, 0.0, "alu"),
    }


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, one launch) of a kernel
# from an ncu capture of this workload, with a hash of the sources it was built from;
# a kernel whose sources changed since the capture reports null.
NCU_TRAFFIC = {
    ("gdn_fwd_fused_tc", "l27b_bf16"): (855.956736e6, "7110374e20a63bf8"),
    ("gdn_fwd_out_tc", "l27b_bf16"): (119.532544e6, "7110374e20a63bf8"),
    ("gdn_bwd_fused_tc", "l27b_bf16"): (936.749056e6, "dc15850ee8e949dc"),
}
KERNEL_SOURCES = {
    "gdn_fwd_fused_tc": ("gdn_tc_fwd.cu", "gdn_tc.cuh", "umma.cuh", "gdn_device.cuh",
                         "gdn_internal.cuh"),
    "gdn_fwd_out_tc": ("gdn_tc_fwd.cu", "gdn_tc.cuh", "umma.cuh", "gdn_device.cuh",
                       "gdn_internal.cuh"),
    "gdn_bwd_fused_tc": ("gdn_tc_bwd.cu", "gdn_tc.cuh", "umma.cuh", "gdn_device.cuh",
                         "gdn_internal.cuh"),
}


def measured_traffic(kernel, workload):
    import hashlib
    entry = NCU_TRAFFIC.get((kernel, workload))
    if entry is None or kernel not in KERNEL_SOURCES:
        return None
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_deltanet_backward_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return entry[0] if h.hexdigest()[:16] == entry[1] else None


def kernel_roofline(b, f, unit, avg_s, pk):
    """Per-kernel diagnostic: the roof (HBM bytes or FLOPs at the unit's peak) that bounds
    the kernel's implementation bytes (kernel_models) and FLOPs, and the achieved rate."""
    peak_alu = alu_fp32_tflops(pk["sm_max_mhz"])
    t_mem = b / (pk["hbm_gbs"] * 1e9)
    peak_c = peak_alu if unit == "alu" else pk["bf16_tflops"]
    t_cmp = f / (peak_c * 1e12)
    if t_cmp > t_mem:
        roof = {"bound": unit, "achieved": f / avg_s / 1e12, "peak": peak_c, "unit": "TFLOP/s"}
        roof["peak_source"] = ("derived: 152 SMs x 128 FP32 lanes x 2 x %.0f MHz" %
                               pk["sm_max_mhz"]) if unit == "alu" else pk["source"] + " bf16"
    else:
        roof = {"bound": "hbm", "achieved": b / avg_s / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "peak_source": pk["source"] + " HBM"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["implementation_bytes"] = b
    roof["flops"] = f
    return roof


def pass_roofline(per, steps, pm, pk, workload):
    """Roofline entry of the dominant pass (forward or backward) of the step: its
    algorithmic bytes and FLOPs (path_model, fp32 chunk-start states) over the average
    per-step time of its kernels (the library's CUDA events on the launch stream).  A
    fused pass is one launch, so this is that kernel's roofline; `traffic` is the ncu
    DRAM bytes of the same launch when the capture matches the current sources."""
    t_pass = {}
    for which, names in (("forward", FWD_KERNELS), ("backward", BWD_KERNELS)):
        t_pass[which] = sum(sum(per.get(n, [])) for n in names) * 1e-3 / steps
    which = max(t_pass, key=t_pass.get)
    names = FWD_KERNELS if which == "forward" else BWD_KERNELS
    launched = [n for n in names if n in per]
    dom = max(launched, key=lambda n: sum(per[n]))
    b = pm["bytes_fwd" if which == "forward" else "bytes_bwd"]
    f = pm["flops_fwd" if which == "forward" else "flops_bwd"]
    t_mem, t_cmp = b / (pk["hbm_gbs"] * 1e9), f / (pk["bf16_tflops"] * 1e12)
    t = t_pass[which]
    if t_cmp > t_mem:
        roof = {"bound": "tensor", "achieved": f / t / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "peak_source": pk["source"] + " bf16 burst"}
    else:
        roof = {"bound": "hbm", "achieved": b / t / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": pk["source"] + " HBM"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    fused = len(launched) == 1 or dom.endswith("_fused_tc")
    traffic = measured_traffic(dom, workload) if fused else None
    roof.update({
        "traffic": traffic, "traffic_over_algorithmic": (traffic / b) if traffic else None,
        "kernel": dom, "pass": which, "pass_kernels": launched,
        "pass_us": t * 1e6, "algorithmic_bytes": b, "algorithmic_flops": f,
        "tensor_frac": (f / t / 1e12) / pk["bf16_tflops"],
        "model": "method bytes per token: q, k, v, alpha, beta_raw, o (forward), dO, dq, dk, "
                 "dv, dalpha, dbeta_raw (backward) and fp32 chunk-start states written once "
                 "and read once, plus the N Hv Dk Dv fp32 boundary states"})
    return roof


# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(index), "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in rows:
            if len(row) < 9:
                continue
            try:
                mhz.append(float(row[1]))
                mx.append(float(row[2]))
            except ValueError:
                continue
            for name, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(mhz)}


# ----------------------------------------------------------------------------
def workload_config(wl, world):
    """The `config` object both arms print for the workload (the reference arm adds its
    per-step sample)."""
    T, N = wl.total_tokens, wl.n_seqs
    return {"workload": "%s: %d x %d tokens, Hk=%d, Hv=%d, Dk=%d, Dv=%d, %s q/k/v/o/dO, "
                        "fp32 gates/state" % (wl.name, N, T // max(N, 1), wl.Hk, wl.Hv, wl.Dk,
                                               wl.Dv, wl.dtype),
            "tokens_per_gpu": T, "io_dtype": wl.dtype,
            "parallelism": "independent batch per GPU" if world > 1 else "single GPU"}


def max_over_ranks(x, world, device):
    """The largest of every rank's x (every rank calls it): the whole job is as slow as its
    slowest rank."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch
    import gated_deltanet_backward_gb300 as gdn

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = W.get(args.workload)
    inp = W.generate(wl)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T, Hk, Hv, Dk, Dv, N = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv, wl.n_seqs

    def dev(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device, dt)

    qkv = dev(inp.qkv, tdt)
    if qkv is not None:   # packed projection rows: q, k, v are strided views
        q, k, v = qkv[:, :Hk * Dk], qkv[:, Hk * Dk:2 * Hk * Dk], qkv[:, 2 * Hk * Dk:]
    else:
        q, k, v = dev(inp.q, tdt), dev(inp.k, tdt), dev(inp.v, tdt)
    alpha, beta_raw = dev(inp.alpha), dev(inp.beta_raw)
    a_log, dt_bias = dev(inp.a_log), dev(inp.dt_bias)
    S0, dS_T, dO = dev(inp.S0), dev(inp.dS_T), dev(inp.dO, tdt)
    layer = gdn.Layer.create(Hk, Hv, Dk, Dv, inp.cu_seqlens, wl.dtype, wl.scale_value(),
                             device=device)
    o = torch.empty(T, Hv * Dv, device=device, dtype=tdt)
    S_T = torch.empty(N, Hv, Dk, Dv, device=device)
    dq = torch.empty(T, Hk * Dk, device=device, dtype=tdt)
    dk = torch.empty_like(dq)
    dv = torch.empty(T, Hv * Dv, device=device, dtype=tdt)
    dalpha = torch.empty(T, Hv, device=device)
    dbeta = torch.empty(T, Hv, device=device)
    da_log = torch.empty(Hv, device=device)
    ddt = torch.empty(Hv, device=device)
    dS0 = torch.empty(N, Hv, Dk, Dv, device=device)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)

    def fwd_on(st):
        layer.forward(q, k, v, alpha, beta_raw, a_log, dt_bias, S0, o, S_T, st, train=True)

    def bwd_on(st):
        layer.backward(q, k, v, alpha, beta_raw, a_log, dt_bias, S0, dO, dS_T, dq, dk, dv,
                       dalpha, dbeta, da_log, ddt, dS0, st, train=True)

    def fwd():
        fwd_on(stream)

    def bwd():
        bwd_on(stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
        flush()
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(layer.ws_bwd) == 0

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    prof = gdn.gdn_profile(max_launches=16 * K)
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with prof:
        for i in range(K):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
            flush()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    f_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    b_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    plain_ms = max_over_ranks(sum(f_ms[i] + b_ms[i] for i in range(K)) / K, world, device)
    # The headline: the same step replayed as two CUDA graphs (forward, backward), which
    # is how a fixed-shape training loop runs it: no per-launch host work or launch gaps,
    # and no profiling events between the kernels.  The plain calls above give the
    # per-kernel times.
    graphed = graph_step_times(fwd_on, bwd_on, flush, K, device, world)
    assert gdn.gdn_read_device_status(layer.ws_bwd) == 0
    if graphed is not None:
        step_ms, f_avg, b_avg = graphed
    else:
        step_ms, f_avg, b_avg = plain_ms, sum(f_ms) / K, sum(b_ms) / K
    value = world * T / (step_ms * 1e-3)

    # per-kernel durations from the profiling hook
    per = {}
    for name, ms in prof.launches():
        per.setdefault(name, []).append(ms)
    launches = prof.count
    tot = sum(sum(v) for v in per.values())
    kernels = {n: {"launches": len(v), "avg_us": 1e3 * sum(v) / len(v),
                   "share": sum(v) / tot if tot else 0.0} for n, v in per.items()}
    pk = _peaks()
    models = kernel_models(wl)
    pm = path_model(wl)
    roof = pass_roofline(per, K, pm, pk, wl.name)
    for name in kernels:
        kb, kf, ku = models[name]
        r = kernel_roofline(kb, kf, ku, kernels[name]["avg_us"] * 1e-6, pk)
        kernels[name].update(implementation_bytes=kb, implementation_frac=r["frac"],
                             implementation_bound=r["bound"])
    t_roof = max(pm["bytes"] / (pk["hbm_gbs"] * 1e9), pm["flops"] / (pk["bf16_tflops"] * 1e12))
    path_roof = {"bytes_per_step": pm["bytes"], "flops_per_step": pm["flops"],
                 "bytes_per_token": pm["bytes_per_token"],
                 "flops_per_token": pm["flops_per_token"],
                 "roofline_us": t_roof * 1e6, "roofline_tokens_per_s": T / t_roof,
                 "frac": (T / (step_ms * 1e-3)) / (T / t_roof),
                 "bound": "hbm" if pm["bytes"] / (pk["hbm_gbs"] * 1e9) >= pm["flops"] / (
                     pk["bf16_tflops"] * 1e12) else "tensor",
                 "peak_source": pk["source"]}

    bf16_states = None
    if wl.dtype == "bf16" and min(Dk, Dv) >= 64 and not args.no_variants:
        # the same step with the chunk-start states kept as bf16 tiles
        # (GDN_FLAG_BF16_SAVED_STATES): same gradients, half the largest byte stream
        layer_b = gdn.Layer.create(Hk, Hv, Dk, Dv, inp.cu_seqlens, wl.dtype, wl.scale_value(),
                                   device=device, bf16_states=True)

        def step_b_on(st):
            layer_b.forward(q, k, v, alpha, beta_raw, a_log, dt_bias, S0, o, S_T, st,
                            train=True)
            layer_b.backward(q, k, v, alpha, beta_raw, a_log, dt_bias, S0, dO, dS_T, dq, dk, dv,
                             dalpha, dbeta, da_log, ddt, dS0, st, train=True)

        def step_b():
            step_b_on(stream)

        for _ in range(args.warmup):
            step_b()
            flush()
        torch.cuda.synchronize()
        gb = graph_step_times(step_b_on, None, flush, K, device, world)
        if gb is not None:
            ms_b = gb[0]
        else:
            evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K)]
            for e0, e1 in evb:
                e0.record(stream)
                step_b()
                e1.record(stream)
                flush()
            torch.cuda.synchronize()
            ms_b = max_over_ranks(sum(a.elapsed_time(b) for a, b in evb) / K, world, device)
        assert gdn.gdn_read_device_status(layer_b.ws_bwd) == 0
        bf16_states = {"ms_per_step": ms_b, "value": world * T / (ms_b * 1e-3),
                       "unit": "tokens/s",
                       "path_frac": (T / (ms_b * 1e-3)) / (T / t_roof),
                       "note": "GDN_FLAG_BF16_SAVED_STATES: chunk-start states kept as bf16 "
                               "tiles; the same gradients bit for bit; path_frac against the "
                               "same method bytes (fp32 states)"}
        del layer_b

    e2e = run_e2e(args, inp, layer, device, tdt, world) if not args.no_e2e else None
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {**workload_config(wl, world),
                   "compute": ("tcgen05 bf16 MMA, fp32 accumulate and state" if wl.dtype == "bf16"
                               else "fp32 CUDA-core FMA"),
                   "l2": "flushed between timed steps: 256 MB write, then 256 MB read",
                   "step": "training step: the forward keeps its chunk operands for the "
                           "backward (GDN_FLAG_KEEP_FOR_BACKWARD / GDN_FLAG_REUSE_FORWARD)",
                   },
        "fwd_ms": f_avg, "bwd_ms": b_avg,
        "ms_per_step_plain": plain_ms,
        "timing": ("CUDA events around K steps replayed as CUDA graphs (forward, backward), "
                   "L2 flush between steps; kernels from the same calls made one by one with "
                   "the library's profiling events (ms_per_step_plain)"
                   if graphed is not None else
                   "CUDA events around K steps of plain calls, L2 flush between steps"),
        "roofline": roof, "path_roofline": path_roof, "kernels": kernels,
        "gpu_launches": launches, "clocks": clocks, "e2e": e2e,
        "bf16_saved_states": bf16_states,
    }
    if rank == 0 and world == 1 and not args.no_decode:
        result["decode"] = run_decode(wl, device, pk)
    if rank == 0 and world == 1 and not args.no_layer_steps:
        result["layer_steps"] = run_layer_steps(wl, device, pk)
    if rank == 0 and world == 1 and not args.no_decode:
        result["kda"] = run_kda(wl, device, pk)
    if rank == 0 and world == 1 and not args.no_context_parallel:
        result["context_parallel"] = run_context_parallel(wl, device, step_ms)
        result["context_parallel_long"] = run_context_parallel(wl, device, None, segments=8,
                                                               tokens=16 * wl.total_tokens)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_tokens)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_decode(wl, device, pk, n_seqs=64, steps=50, warmup=5):
    """gdn_decode_step on a batch of n_seqs sequences with the workload's head shape:
    one new token per sequence per step, the fp32 state updated in place (its
    n_seqs * Hv * Dk * Dv * 4 bytes, read and written once a step, exceed the L2, so
    no flush is needed).  Synthetic inputs, resident on the device."""
    import torch
    import gated_deltanet_backward_gb300 as gdn
    Hk, Hv, Dk, Dv = wl.Hk, wl.Hv, wl.Dk, wl.Dv
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device).manual_seed(1234)
    rn = lambda *sh, dt=torch.float32: torch.randn(*sh, generator=g, device=device).to(dt)
    q, k = rn(n_seqs, Hk * Dk, dt=td), rn(n_seqs, Hk * Dk, dt=td)
    v, o = rn(n_seqs, Hv * Dv, dt=td), torch.empty(n_seqs, Hv * Dv, device=device, dtype=td)
    alpha, beta_raw = rn(n_seqs, Hv), rn(n_seqs, Hv)
    a_log = torch.rand(Hv, generator=g, device=device) * 2 - 1
    dt_bias = rn(Hv) * 0.1
    S = rn(n_seqs, Hv, Dk, Dv) * 0.1
    shape = gdn.make_shape(Hk, Hv, Dk, Dv, n_seqs, n_seqs, n_seqs, wl.dtype, 0.0)
    step = lambda: gdn.gdn_decode_step(shape, q, k, v, alpha, beta_raw, a_log, dt_bias, S, S, o)
    for _ in range(warmup):
        step()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / steps
    state_bytes = 2 * n_seqs * Hv * Dk * Dv * 4
    io_bytes = n_seqs * ((2 * Hk * Dk + 2 * Hv * Dv) * (2 if wl.dtype == "bf16" else 4) + 8 * Hv)
    gbs = (state_bytes + io_bytes) / (us * 1e-6) / 1e9
    return {"n_seqs": n_seqs, "us_per_step": us, "tokens_per_s": n_seqs / (us * 1e-6),
            "bytes_per_step": state_bytes + io_bytes, "achieved_gbs": gbs,
            "frac": gbs / pk["hbm_gbs"], "bound": "hbm",
            "note": "gdn_decode_step, one token per sequence, state in place; "
                    "value head shape of the workload"}


def run_layer_steps(wl, device, pk, K=4, eps=1e-6, steps=10, warmup=3):
    """The layer steps either side of the recurrence at the workload's layer shape: the
    causal conv1d + SiLU over the packed q|k|v rows (C = 2 Hk Dk + Hv Dv channels, kernel
    K) and the gated RMSNorm over the Hv heads of o, forward and backward (weight
    gradients included).  Each kernel is timed alone with CUDA events around its own
    launch, after an L2 flush (L2Flush); bytes are the algorithmic ones
    (every operand read once, every result written once).  Synthetic inputs (N(0, 1)
    activations, conv weights U(-0.05, 0.05), norm weights U(0.9, 1.1)), resident."""
    import torch
    import gated_deltanet_backward_gb300 as gdn
    T, Hk, Hv, Dk, Dv = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv
    C, Wd = 2 * Hk * Dk + Hv * Dv, Hv * Dv
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    es = 2 if wl.dtype == "bf16" else 4
    g = torch.Generator(device=device).manual_seed(4321)
    rn = lambda *sh: torch.randn(*sh, generator=g, device=device).to(td)
    x, dyc = rn(T, C), rn(T, C)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    w = (torch.rand(C, K, generator=g, device=device) * 2 - 1) * 0.05
    dw = torch.empty_like(w)
    o, z, dyn = rn(T, Wd), rn(T, Wd), rn(T, Wd)
    yn, d_o, dz = torch.empty_like(o), torch.empty_like(o), torch.empty_like(o)
    gamma = 0.9 + 0.2 * torch.rand(Dv, generator=g, device=device)
    dg = torch.empty_like(gamma)
    cu_h = np.asarray([0] + list(np.cumsum(wl.seqlens)), dtype=np.int32)
    cu = torch.from_numpy(cu_h).to(device)
    ws_c = torch.empty(max(256, gdn.gdn_conv1d_silu_workspace_bytes(T, C, K)), dtype=torch.uint8,
                       device=device)
    ws_n = torch.empty(gdn.gdn_gated_rmsnorm_workspace_bytes(Dv), dtype=torch.uint8,
                       device=device)
    flush = L2Flush(device)
    calls = {
        "conv1d_silu_fwd": (lambda: gdn.gdn_conv1d_silu_forward(x, w, cu, y),
                            2 * T * C * es + C * K * 4),
        "conv1d_silu_bwd": (lambda: gdn.gdn_conv1d_silu_backward(x, w, cu, dyc, dx, dw, ws_c),
                            3 * T * C * es + 2 * C * K * 4),
        "gated_rmsnorm_fwd": (lambda: gdn.gdn_gated_rmsnorm_forward(o, z, gamma, yn, eps),
                              3 * T * Wd * es + Dv * 4),
        "gated_rmsnorm_bwd": (lambda: gdn.gdn_gated_rmsnorm_backward(o, z, gamma, dyn, d_o, dz,
                                                                     eps, dg, ws_n),
                              5 * T * Wd * es + 2 * Dv * 4),
    }
    stream = torch.cuda.current_stream()
    out = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        prof = gdn.gdn_profile(max_launches=4 * steps)
        torch.cuda.synchronize()
        with prof:
            for e0, e1 in ev:
                flush()
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        call_us = 1e3 * sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
        # the library's events around each of its launches (the kernels alone)
        us = 1e3 * sum(ms for _, ms in prof.launches()) / steps
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us": us, "call_us": call_us, "bytes": nbytes, "achieved_gbs": gbs,
                     "frac": gbs / pk["hbm_gbs"], "bound": "hbm",
                     "kernels": sorted({k for k, _ in prof.launches()})}
    out["shape"] = {"tokens": T, "channels": C, "kernel_size": K, "heads": Hv, "head_dim": Dv,
                    "dtype": wl.dtype}
    out["note"] = ("each call timed alone after an L2 flush: us = the library's CUDA events "
                   "around its launches (the weight-gradient partial sums of the backward "
                   "calls included), call_us = events around the whole Python call")
    return out


def run_kda(wl, device, pk, n_seqs=64, prefill_tokens=1024, steps=20, warmup=3):
    """The KDA variant (a decay gate per key channel) with the workload's head shape:
    gdn_kda_forward as a decode step on n_seqs one-token sequences (state in place; bytes
    as for the decode step plus the per-channel gate rows) against HBM, and as a prefill
    of one prefill_tokens-token sequence in token form (tokens/s), and that prefill's
    training step (gdn_kda_forward + gdn_kda_backward).  Synthetic inputs."""
    import torch
    import gated_deltanet_backward_gb300 as gdn
    Hk, Hv, Dk, Dv = wl.Hk, wl.Hv, wl.Dk, wl.Dv
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    es = 2 if wl.dtype == "bf16" else 4
    g = torch.Generator(device=device).manual_seed(77)
    rn = lambda *sh, dt=torch.float32: torch.randn(*sh, generator=g, device=device).to(dt)
    a_log = torch.rand(Hv, generator=g, device=device) * 2 - 1
    b_alpha = rn(Hv * Dk) * 0.1
    out = {}
    for name, N, T in (("decode", n_seqs, n_seqs), ("prefill", 1, prefill_tokens)):
        q, k, v = rn(T, Hk * Dk, dt=td), rn(T, Hk * Dk, dt=td), rn(T, Hv * Dv, dt=td)
        alpha, beta = rn(T, Hv * Dk), rn(T, Hv)
        o = torch.empty(T, Hv * Dv, device=device, dtype=td)
        S = rn(N, Hv, Dk, Dv) * 0.1
        cu = (torch.arange(N + 1, device=device, dtype=torch.int32) if name == "decode"
              else torch.tensor([0, T], device=device, dtype=torch.int32))
        shape = gdn.make_shape(Hk, Hv, Dk, Dv, N, 0, T, wl.dtype, 0.0)
        step = lambda: gdn.gdn_kda_forward(shape, q, k, v, alpha, beta, a_log, b_alpha, cu, S, S,
                                           o)
        n_steps = steps if name == "decode" else 2
        for _ in range(warmup if name == "decode" else 1):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / n_steps
        entry = {"sequences": N, "tokens": T, "us_per_call": us,
                 "tokens_per_s": T / (us * 1e-6)}
        if name == "decode":
            nbytes = (2 * N * Hv * Dk * Dv * 4 + N * (2 * Hk * Dk + 2 * Hv * Dv) * es
                      + N * Hv * (Dk + 1) * 4)
            gbs = nbytes / (us * 1e-6) / 1e9
            entry.update({"bytes_per_call": nbytes, "achieved_gbs": gbs,
                          "frac": gbs / pk["hbm_gbs"], "bound": "hbm"})
        else:
            entry["note"] = "token form: one token after another per (value head, column slice)"
            # the training step of the same prefill: forward, then gdn_kda_backward
            dO = rn(T, Hv * Dv, dt=td)
            dS_T = rn(N, Hv, Dk, Dv) * 0.1
            S0 = rn(N, Hv, Dk, Dv) * 0.1
            dq, dk = torch.empty_like(q), torch.empty_like(k)
            dv = torch.empty_like(v)
            dalpha, dbeta = torch.empty_like(alpha), torch.empty_like(beta)
            da_log, db_al = torch.empty_like(a_log), torch.empty_like(b_alpha)
            dS0 = torch.empty_like(S0)
            ws = torch.empty(gdn.gdn_kda_backward_workspace_bytes(shape), dtype=torch.uint8,
                             device=device)
            S_T = torch.empty_like(S0)

            def train():
                gdn.gdn_kda_forward(shape, q, k, v, alpha, beta, a_log, b_alpha, cu, S0, S_T, o)
                gdn.gdn_kda_backward(shape, q, k, v, alpha, beta, a_log, b_alpha, cu, S0, dO,
                                     dS_T, dq, dk, dv, dalpha, dbeta, da_log, db_al, dS0, ws)

            train()
            torch.cuda.synchronize()
            e0.record()
            for _ in range(2):
                train()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 2
            entry["training_step_ms"] = ms
            entry["training_tokens_per_s"] = T / (ms * 1e-3)
            # the same prefill chunked on the tensor cores (gdn_kda_forward_chunked)
            if wl.dtype == "bf16" and Dk in (64, 128) and Dv in (64, 128):
                off, NC = gdn.gdn_plan(np.array([0, T], dtype=np.int32))
                shape_c = gdn.make_shape(Hk, Hv, Dk, Dv, N, NC, T, wl.dtype, 0.0)
                coff = torch.from_numpy(off).to(device)
                wsc = torch.empty(gdn.gdn_kda_forward_chunked_workspace_bytes(shape_c),
                                  dtype=torch.uint8, device=device)

                def chunked():
                    gdn.gdn_kda_forward_chunked(shape_c, q, k, v, alpha, beta, a_log, b_alpha, cu,
                                                coff, S0, S_T, o, wsc)

                chunked()
                torch.cuda.synchronize()
                e0.record()
                for _ in range(steps):
                    chunked()
                e1.record()
                torch.cuda.synchronize()
                us_c = 1e3 * e0.elapsed_time(e1) / steps
                entry["chunked"] = {"us_per_call": us_c, "tokens_per_s": T / (us_c * 1e-6),
                                    "note": "gdn_kda_forward_chunked: the chunk algebra, "
                                            "products, walk and output on the tensor cores"}
        out[name] = entry
    return out


def run_context_parallel(wl, device, plain_step_ms, segments=4, steps=3, warmup=1, tokens=None):
    """One sequence of the workload's length (or `tokens`) cut into `segments` equal
    segments, all on this GPU (context parallelism run serially): the whole segmented
    training step (segment maps, scans, final passes) and each pass alone, with CUDA
    events.  per_rank_ms adds up the passes one rank of a `segments`-GPU group would run
    (exchange not included).  With `tokens` the unsegmented step on the whole sequence is
    timed too (plain_step_ms).  Synthetic inputs, resident."""
    import torch
    from gated_deltanet_backward_gb300 import context_parallel as cp
    T, Hk, Hv, Dk, Dv = tokens or wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv
    td = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device).manual_seed(99)
    rn = lambda *sh, dt=torch.float32: torch.randn(*sh, generator=g, device=device).to(dt)
    L = T // segments
    a_log = torch.rand(Hv, generator=g, device=device) * 2 - 1
    dt_bias = rn(Hv) * 0.1
    segs = [cp.Segment(rn(L, Hk * Dk, dt=td), rn(L, Hk * Dk, dt=td), rn(L, Hv * Dv, dt=td),
                       rn(L, Hv), rn(L, Hv), a_log, dt_bias) for _ in range(segments)]
    dOs = [rn(L, Hv * Dv, dt=td) for _ in range(segments)]
    S0, dS_T = rn(1, Hv, Dk, Dv) * 0.1, rn(1, Hv, Dk, Dv) * 0.1
    ops = cp.GpuSegmentOps(Hk, Hv, Dk, Dv, wl.dtype)
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            out = fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n, out

    def step():
        outs, S_T, ctx = cp.forward(ops, segs, S0)
        return cp.backward(ops, segs, ctx, dOs, dS_T)

    step_ms, _ = timed(step, steps)
    if tokens:
        whole = cp.Segment(torch.cat([sg.q for sg in segs]), torch.cat([sg.k for sg in segs]),
                           torch.cat([sg.v for sg in segs]), torch.cat([sg.alpha for sg in segs]),
                           torch.cat([sg.beta_raw for sg in segs]), a_log, dt_bias)
        dO_all = torch.cat(dOs)

        def plain():
            ops.forward(whole, S0, keep=True)
            return ops.backward(whole, S0, dO_all, dS_T)

        plain_step_ms, _ = timed(plain, steps)
        del whole
    s0 = segs[0]
    map_ms, Phi = timed(lambda: ops.state_map(s0), steps)
    fz_ms, _ = timed(lambda: ops.forward(s0, None, keep=False), steps)
    fwd_ms, _ = timed(lambda: ops.forward(s0, S0, keep=True), steps)
    bwd_ms, _ = timed(lambda: ops.backward(s0, S0, dOs[0], dS_T), steps)
    comp_ms, _ = timed(lambda: ops.compose(Phi, S0, S0, False), steps)
    per_rank = map_ms + fz_ms + fwd_ms + 2 * bwd_ms + 2 * (segments - 1) * comp_ms
    return {"segments": segments, "tokens_per_segment": L, "one_gpu_step_ms": step_ms,
            "plain_step_ms": plain_step_ms,
            "segment_pass_ms": {"state_map": map_ms, "forward_from_zero": fz_ms,
                                "forward": fwd_ms, "backward": bwd_ms, "compose": comp_ms},
            "per_rank_ms": per_rank,
            "note": "per_rank_ms: the passes one rank of a %d-GPU group runs (state map, "
                    "forward from zero, forward, 2 backwards, 2 scans), measured here one "
                    "by one; the all-gathers are not included" % segments}


def run_e2e(args, inp, layer, device, tdt, world):
    """Same metric through the public API with host buffers: every step copies all its
    inputs from pinned host memory to the device and reads all its results (o, S_T and
    every gradient) back into pinned host memory.  The steps are pipelined over three
    streams, as a training loop feeding a GPU from the host would run them: step i's
    uploads (one copy stream) overlap step i-1's compute, its downloads (another copy
    stream) overlap step i+1's compute; device inputs and outputs are double-buffered and
    ordered by events.  value = K steps' tokens / the time from the first upload to the
    last download; serial_ms_per_step is the same steps on one stream, nothing overlapped."""
    import torch
    wl = inp.wl
    T, Hk, Hv, Dk, Dv, N = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv, wl.n_seqs

    def pin(a, dt=torch.float32):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dt).pin_memory()

    packed = inp.qkv is not None
    qkv_rows = inp.qkv if packed else np.concatenate([inp.q, inp.k, inp.v], axis=1)
    h_in = dict(qkv=pin(qkv_rows, tdt), alpha=pin(inp.alpha), beta_raw=pin(inp.beta_raw),
                a_log=pin(inp.a_log), dt_bias=pin(inp.dt_bias), dO=pin(inp.dO, tdt),
                S0=pin(inp.S0), dS_T=pin(inp.dS_T))
    outs = dict(o=(T, Hv * Dv, tdt), dq=(T, Hk * Dk, tdt), dk=(T, Hk * Dk, tdt),
                dv=(T, Hv * Dv, tdt), dalpha=(T, Hv, torch.float32),
                dbeta=(T, Hv, torch.float32), da_log=(Hv, None, torch.float32),
                ddt=(Hv, None, torch.float32), S_T=(N, Hv * Dk * Dv, torch.float32),
                dS0=(N, Hv * Dk * Dv, torch.float32))

    def dev_in():
        return {k: (None if v is None else torch.empty(v.shape, dtype=v.dtype, device=device))
                for k, v in h_in.items()}

    def dev_out():
        return {k: torch.empty(s[:2] if s[1] else (s[0],), dtype=s[2], device=device)
                for k, s in outs.items()}

    d_in, d_out = [dev_in(), dev_in()], [dev_out(), dev_out()]
    h_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in d_out[0].items()}
             for _ in range(2)]
    bytes_in = sum(v.numel() * v.element_size() for v in h_in.values() if v is not None)
    bytes_out = sum(v.numel() * v.element_size() for v in h_out[0].values())

    def compute(di, do, st):
        qkv = di["qkv"]
        q, k, v = qkv[:, :Hk * Dk], qkv[:, Hk * Dk:2 * Hk * Dk], qkv[:, 2 * Hk * Dk:]
        layer.forward(q, k, v, di["alpha"], di["beta_raw"], di["a_log"], di["dt_bias"], di["S0"],
                      do["o"], do["S_T"].view(N, Hv, Dk, Dv), st, train=True)
        layer.backward(q, k, v, di["alpha"], di["beta_raw"], di["a_log"], di["dt_bias"],
                       di["S0"], di["dO"], di["dS_T"], do["dq"], do["dk"], do["dv"], do["dalpha"],
                       do["dbeta"], do["da_log"], do["ddt"], do["dS0"].view(N, Hv, Dk, Dv), st,
                       train=True)

    def upload(di):
        for key, h in h_in.items():
            if h is not None:
                di[key].copy_(h, non_blocking=True)

    def download(do, ho):
        for key, h in ho.items():
            h.copy_(do[key], non_blocking=True)

    s_up, s_cmp, s_down = (torch.cuda.Stream(device) for _ in range(3))

    def pipelined(K):
        ev_up = [torch.cuda.Event() for _ in range(K)]
        ev_cmp = [torch.cuda.Event() for _ in range(K)]
        ev_down = [torch.cuda.Event() for _ in range(K)]
        for i in range(K):
            b = i % 2
            if i >= 2:
                s_up.wait_event(ev_cmp[i - 2])    # step i-2's compute has read d_in[b]
            with torch.cuda.stream(s_up):
                upload(d_in[b])
            ev_up[i].record(s_up)
            s_cmp.wait_event(ev_up[i])
            if i >= 2:
                s_cmp.wait_event(ev_down[i - 2])  # step i-2's downloads have read d_out[b]
            compute(d_in[b], d_out[b], s_cmp)
            ev_cmp[i].record(s_cmp)
            s_down.wait_event(ev_cmp[i])
            with torch.cuda.stream(s_down):
                download(d_out[b], h_out[b])
            ev_down[i].record(s_down)

    def serial(K):
        st = torch.cuda.current_stream(device)
        for _ in range(K):
            upload(d_in[0])
            compute(d_in[0], d_out[0], st)
            download(d_out[0], h_out[0])

    K = args.steps
    res = {}
    for name, fn, first in (("serial", serial, None), ("pipelined", pipelined, s_up)):
        fn(max(2, args.warmup))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(first or torch.cuda.current_stream(device))
        fn(K)
        e1.record(s_down if first else torch.cuda.current_stream(device))
        torch.cuda.synchronize()
        res[name] = max_over_ranks(e0.elapsed_time(e1) / K, world, device)
    assert gdn_status_ok(layer)
    ms = res["pipelined"]
    return {"value": world * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "serial_ms_per_step": res["serial"], "h2d_bytes_per_step": int(bytes_in),
            "d2h_bytes_per_step": int(bytes_out),
            "pipeline": "3 streams (upload, compute, download), double-buffered device I/O"}


def gdn_status_ok(layer):
    import gated_deltanet_backward_gb300 as gdn
    return gdn.gdn_read_device_status(layer.ws_bwd) == 0


def _oracle_step(inp, tokens, n_threads=0):
    import oracle
    wl = inp.wl
    cu = np.array([0, tokens], np.int32) if tokens < wl.total_tokens else inp.cu_seqlens
    sl = slice(0, tokens)
    S0 = inp.S0 if tokens >= wl.total_tokens else (None if inp.S0 is None else inp.S0[:1])
    dS_T = inp.dS_T if tokens >= wl.total_tokens else (None if inp.dS_T is None else inp.dS_T[:1])
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, scale=wl.scale_value(),
              n_threads=n_threads)
    oracle.forward(inp.q[sl], inp.k[sl], inp.v[sl], inp.alpha[sl], inp.beta_raw[sl], inp.a_log,
                   inp.dt_bias, cu, S0, **kw)
    oracle.backward(inp.q[sl], inp.k[sl], inp.v[sl], inp.alpha[sl], inp.beta_raw[sl], inp.a_log,
                    inp.dt_bias, cu, inp.dO[sl], S0, dS_T, **kw)


def cpu_baseline(wl, inp, tokens, one_thread_tokens=256):
    """The oracle (f64, token by token) on the host cores: the whole workload (up to
    `tokens` tokens) on every hardware thread, and a shorter sample on one thread."""
    import oracle
    tokens = min(tokens, wl.total_tokens)
    t0 = time.perf_counter()
    _oracle_step(inp, tokens)
    dt = time.perf_counter() - t0
    out = {"value": tokens / dt, "unit": "tokens/s", "cores": oracle.hardware_threads(),
           "kind": "oracle",
           "sample": "f64 token-by-token forward + backward of the first %d tokens of %s "
                     "(all %d value heads), one pass, %.1f s" % (tokens, wl.name, wl.Hv, dt)}
    n1 = min(one_thread_tokens, wl.total_tokens)
    if n1 > 0:
        t0 = time.perf_counter()
        _oracle_step(inp, n1, n_threads=1)
        dt1 = time.perf_counter() - t0
        out["one_thread"] = {"value": n1 / dt1, "unit": "tokens/s", "cores": 1,
                             "sample": "the first %d tokens, one pass, %.1f s" % (n1, dt1)}
    return out


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return
    import oracle
    wl = W.get(args.workload)
    inp = W.generate(wl)
    tokens = min(args.ref_tokens, wl.total_tokens)
    oracle.build()
    for _ in range(args.warmup):
        _oracle_step(inp, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(inp, tokens)
    dt = (time.perf_counter() - t0) / args.steps
    value = tokens / dt
    sample = ("f64 token-by-token CPU oracle, forward + backward of %s of %s (all %d value "
              "heads) per step" % ("all %d tokens" % tokens if tokens == wl.total_tokens else
                                   "the first %d tokens" % tokens, wl.name, wl.Hv))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {**workload_config(wl, world),
                   "sample_tokens_per_step": tokens,
                   "compute": "f64 token-by-token CPU oracle on the host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.hardware_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="l27b_bf16", choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=4096)
    ap.add_argument("--ref-tokens", type=int, default=4096)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-context-parallel", action="store_true",
                    help="skip the context-parallel (segmented sequence) measurement")
    ap.add_argument("--no-layer-steps", action="store_true",
                    help="skip the conv1d + SiLU / gated RMSNorm measurement")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the step with bf16 chunk-start states")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
