"""Test harness: runs the CUDA library and the CPU oracle on one seeded draw.

Not collected by pytest (no ``test_`` prefix).  The CUDA side goes through the
Python binding of the C ABI; the oracle side through ``oracle``.  Both consume
the same ``workloads.Inputs`` arrays.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

GRADS = ("dq", "dk", "dv", "dalpha", "dbeta_raw", "da_log", "ddt_bias", "dS0")
TOL = {"f32": 1e-3, "bf16": 2e-2}


def rel_err(gpu, ref) -> float:
    """max|gpu - ref| / max|ref|; for an all-zero reference, max|gpu| itself."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(np.abs(gpu).max()) if gpu.size else 0.0
    return float(np.abs(gpu - ref).max() / den)


class DeviceRun:
    """Device copies of one draw plus every output of one forward + backward.

    train=True (the default) runs the pair as a training step: the forward keeps
    the backward's chunk operands and the backward reuses them; train=False has
    each call compute everything itself."""

    def __init__(self, inp: W.Inputs, device="cuda", dense=False, run_backward=True,
                 train=True, bf16_states=False):
        import torch
        import gated_deltanet_backward_gb300 as gdn
        self.inp = inp
        wl = inp.wl
        self.tdtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        T, Hk, Hv, Dk, Dv = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv

        def dev(a, dt=None):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device=device,
                                                                dtype=dt or torch.float32)

        if inp.qkv is not None and not dense:
            self.qkv = dev(inp.qkv, self.tdtype)
            self.q = self.qkv[:, : Hk * Dk]
            self.k = self.qkv[:, Hk * Dk: 2 * Hk * Dk]
            self.v = self.qkv[:, 2 * Hk * Dk:]
        else:
            self.q, self.k, self.v = (dev(x, self.tdtype) for x in (inp.q, inp.k, inp.v))
        self.alpha, self.beta_raw = dev(inp.alpha), dev(inp.beta_raw)
        self.a_log, self.dt_bias = dev(inp.a_log), dev(inp.dt_bias)
        self.S0 = None if inp.S0 is None else dev(inp.S0)
        self.dO = dev(inp.dO, self.tdtype)
        self.dS_T = None if inp.dS_T is None else dev(inp.dS_T)
        self.layer = gdn.Layer.create(Hk, Hv, Dk, Dv, inp.cu_seqlens, wl.dtype,
                                      wl.scale_value(), device=device, head_map=wl.head_map,
                                      bf16_states=bf16_states)
        N = wl.n_seqs
        self.o = torch.full((T, Hv * Dv), float("nan"), device=device, dtype=self.tdtype)
        self.S_T = torch.full((N, Hv, Dk, Dv), float("nan"), device=device)
        self.train = train
        self.grads = None
        self.run_forward()
        if run_backward:
            self.run_backward()

    def run_forward(self):
        """The forward again on the same inputs, into the same o, S_T and saved states."""
        import gated_deltanet_backward_gb300 as gdn
        self.layer.forward(self.q, self.k, self.v, self.alpha, self.beta_raw, self.a_log,
                           self.dt_bias, self.S0, self.o, self.S_T, train=self.train)
        # a training step's backward shares the forward's workspace (and status word)
        self.fwd_status = gdn.gdn_read_device_status(self.layer.ws_bwd) if self.train else None

    def device_outputs(self) -> dict:
        """Every output of the last forward (and backward) as device tensors."""
        out = dict(o=self.o, S_T=self.S_T, saved=self.layer.saved_states)
        if self.grads is not None:
            out.update(self.grads)
        return out

    def run_backward(self, train=None):
        import torch
        train = self.train if train is None else train
        wl = self.inp.wl
        T, Hk, Hv, Dk, Dv, N = wl.total_tokens, wl.Hk, wl.Hv, wl.Dk, wl.Dv, wl.n_seqs
        dev = self.o.device
        nan = float("nan")
        g = dict(dq=torch.full((T, Hk * Dk), nan, device=dev, dtype=self.tdtype),
                 dk=torch.full((T, Hk * Dk), nan, device=dev, dtype=self.tdtype),
                 dv=torch.full((T, Hv * Dv), nan, device=dev, dtype=self.tdtype),
                 dalpha=torch.full((T, Hv), nan, device=dev),
                 dbeta_raw=torch.full((T, Hv), nan, device=dev),
                 da_log=torch.full((Hv,), nan, device=dev),
                 ddt_bias=torch.full((Hv,), nan, device=dev),
                 dS0=torch.full((N, Hv, Dk, Dv), nan, device=dev))
        self.layer.backward(self.q, self.k, self.v, self.alpha, self.beta_raw, self.a_log,
                            self.dt_bias, self.S0, self.dO, self.dS_T, g["dq"], g["dk"], g["dv"],
                            g["dalpha"], g["dbeta_raw"], g["da_log"], g["ddt_bias"], g["dS0"],
                            train=train)
        self.grads = g
        return g

    def status(self, backward=False) -> int:
        import gated_deltanet_backward_gb300 as gdn
        if self.train and not backward:
            return self.fwd_status
        return gdn.gdn_read_device_status(self.layer.ws_bwd if backward else self.layer.ws_fwd)

    def host(self):
        """All outputs as f64 numpy arrays."""
        import torch
        torch.cuda.synchronize()
        out = dict(o=self.o.double().cpu().numpy(), S_T=self.S_T.double().cpu().numpy())
        out["saved"] = saved_states_dense(self.layer.saved_states, self.inp.wl,
                                          self.layer.bf16_states)
        if self.grads is not None:
            for k, v in self.grads.items():
                out[k] = v.double().cpu().numpy()
        return out


def saved_states_dense(saved, wl: W.Workload, bf16_states=False) -> np.ndarray:
    """The saved chunk-start states as [total_chunks, Hv, Dk, Dv] f64, decoded from the
    buffer's documented format (include/gdn.h): fp32 blocks, or with
    GDN_FLAG_BF16_SAVED_STATES bf16 S^T tiles of max(Dv, 64) rows in the
    128-byte-swizzled K-major layout."""
    import torch
    NC, Hv, Dk, Dv = wl.total_chunks, wl.Hv, wl.Dk, wl.Dv
    raw = saved.detach().reshape(-1).view(torch.uint8).cpu().numpy()
    if not bf16_states:
        return raw[:NC * Hv * Dk * Dv * 4].view(np.float32).astype(np.float64).reshape(
            NC, Hv, Dk, Dv)
    MV = max(Dv, 64)
    tile = -(-Dk // 64) * MV * 128
    u16 = raw[:NC * Hv * tile].view(np.uint16).reshape(NC * Hv, tile // 2)
    v = np.arange(Dv)[:, None]
    k = np.arange(Dk)[None, :]
    off = ((k // 64) * MV + v) * 128 + (((k % 64) // 8) ^ (v % 8)) * 16 + (k % 8) * 2
    bits = u16[:, off // 2].astype(np.uint32) << 16          # [NC*Hv, Dv, Dk]
    st = bits.view(np.float32).astype(np.float64).reshape(NC, Hv, Dv, Dk)
    return st.transpose(0, 1, 3, 2)


def head_group_inputs(inp: W.Inputs, kh: int, count: int = 1) -> W.Inputs:
    """The inputs of key heads kh .. kh + count - 1 and their v_repeat value heads each, as
    a stand-alone draw (heads are independent, so the oracle can check some groups of a
    large batch)."""
    wl = inp.wl
    r, Dk, Dv = wl.v_repeat, wl.Dk, wl.Dv
    hs = slice(kh * r, (kh + count) * r)
    sub = W.replace(wl, Hk=count, Hv=r * count, name=wl.name + "_kh%d+%d" % (kh, count))
    return W.Inputs(sub, inp.cu_seqlens, None,
                    inp.q[:, kh * Dk:(kh + count) * Dk], inp.k[:, kh * Dk:(kh + count) * Dk],
                    inp.v[:, kh * r * Dv:(kh + count) * r * Dv], inp.alpha[:, hs],
                    inp.beta_raw[:, hs], inp.a_log[hs], inp.dt_bias[hs],
                    None if inp.S0 is None else inp.S0[:, hs],
                    inp.dO[:, kh * r * Dv:(kh + count) * r * Dv],
                    None if inp.dS_T is None else inp.dS_T[:, hs])


def head_group_outputs(out: dict, wl: W.Workload, kh: int, count: int = 1) -> dict:
    r, Dk, Dv = wl.v_repeat, wl.Dk, wl.Dv
    hs = slice(kh * r, (kh + count) * r)
    vs = slice(kh * r * Dv, (kh + count) * r * Dv)
    ks = slice(kh * Dk, (kh + count) * Dk)
    sel = dict(o=out["o"][:, vs], S_T=out["S_T"][:, hs], saved=out["saved"][:, hs])
    if "dq" in out:
        sel.update(dq=out["dq"][:, ks], dk=out["dk"][:, ks], dv=out["dv"][:, vs],
                   dalpha=out["dalpha"][:, hs], dbeta_raw=out["dbeta_raw"][:, hs],
                   da_log=out["da_log"][hs], ddt_bias=out["ddt_bias"][hs], dS0=out["dS0"][:, hs])
    return sel


def oracle_outputs(inp: W.Inputs, backward=True, n_threads=0) -> dict:
    wl = inp.wl
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, scale=wl.scale_value(),
              n_threads=n_threads, head_map=wl.head_map)
    o, S_T, states = oracle.forward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log,
                                    inp.dt_bias, inp.cu_seqlens, inp.S0, chunk=W.CHUNK, **kw)
    out = dict(o=o, S_T=S_T, saved=states)
    if backward:
        out.update(oracle.backward(inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log,
                                   inp.dt_bias, inp.cu_seqlens, inp.dO, inp.S0, inp.dS_T, **kw))
    return out


def compare(gpu: dict, ref: dict, tol: float, keys=None) -> dict:
    keys = keys or [k for k in ref if k in gpu]
    errs = {k: rel_err(gpu[k], ref[k]) for k in keys}
    for k in keys:
        assert np.all(np.isfinite(gpu[k])), "%s has non-finite values" % k
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, "tensors over tolerance %g: %s (all: %s)" % (tol, bad, errs)
    return errs
