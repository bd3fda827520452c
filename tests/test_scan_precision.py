"""Design check for replacing the sequential chunk walks by a log-depth scan over the
chunks' affine state maps S_next = Phi_c S + R_c (Gated Delta Networks' chunk form;
oracle/chunked.py states the maps and the scan, pinned against the token oracle): formed
with bf16-rounded operands and fp32 accumulation, as the tensor cores' kind::f16 would,
the scan's chunk-start states are no less accurate than those of the sequential walk's
own arithmetic (fp32 state, bf16 operands in X = W S and in the (diag(c) K)^T Delta
update).

One 64-chunk sequence at the head size of the 27B layer (128 x 128), keys, values and
betas drawn as the workloads draw them, and slow gates (0.0005 to 0.05 nats a token),
where every chunk's map carries the state far: the workloads' own gates forget within a
chunk (e^{G_last} ~ e^-50), which makes every method exact to fp32.
"""
import numpy as np
import pytest

import workloads as W
from oracle import chunked

C, N_CHUNKS, D = 64, 64, 128


def _round_bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def _f32(x):
    return np.asarray(x, np.float32)


def _chunks(decay, seed=2):
    wl = W.custom(dtype="bf16", seed=seed, Hk=1, Hv=1, Dk=D, Dv=D, seqlens=(C * N_CHUNKS,),
                  S0_std=0.1, dt_bias_std=0.1)
    inp = W.generate(wl)
    rng = np.random.default_rng(seed)
    maps, parts = [], []
    for c in range(N_CHUNKS):
        s = slice(C * c, C * (c + 1))
        Q, _ = chunked._l2(inp.q[s].astype(np.float64))
        K, _ = chunked._l2(inp.k[s].astype(np.float64))
        V = inp.v[s].astype(np.float64)
        b = chunked.sigmoid(inp.beta_raw[s, 0].astype(np.float64))
        G = np.cumsum(-decay * (1.0 + 0.5 * rng.random(C)))
        maps.append(chunked.chunk_map(Q, K, V, b, G, 1.0))
        _, _, cache = chunked.chunk_forward(Q, K, V, b, G, np.zeros((D, D)), 1.0)
        parts.append((np.exp(G[-1]), cache["cdec"][:, None] * K, cache["W"], cache["U"]))
    return maps, parts, inp.S0[0, 0].astype(np.float64)


def _scan_bf16(maps, S0):
    """Hillis-Steele inclusive scan of the maps, every composition from bf16 operands."""
    pre = [(_f32(P), _f32(R)) for P, R in maps]
    step = 1
    while step < len(pre):
        nxt = list(pre[:step])
        for i in range(step, len(pre)):
            (P2, R2), (P1, R1) = pre[i], pre[i - step]
            P2b = _round_bf16(P2)
            nxt.append((_f32(P2b @ _round_bf16(P1)), _f32(P2b @ _round_bf16(R1)) + R2))
        pre, step = nxt, 2 * step
    S0 = _f32(S0)
    return [S0] + [_f32(_round_bf16(P) @ _round_bf16(S0)) + R for P, R in pre[:-1]]


def _walk_bf16(parts, S0):
    """The sequential walk's arithmetic: fp32 state, bf16 operands in its products."""
    S, out = _f32(S0), [_f32(S0)]
    for a, Kd, Wm, U in parts[:-1]:
        Delta = _f32(U) - _f32(_round_bf16(Wm) @ _round_bf16(S))
        S = _f32(np.float32(a) * S + _f32(_round_bf16(Kd).T @ _round_bf16(Delta)))
        out.append(S)
    return out


def _err(states, ref):
    return max(np.abs(s - r).max() for s, r in zip(states, ref)) / max(np.abs(r).max() for r in ref)


@pytest.mark.parametrize("decay", [0.0005, 0.005, 0.05])
def test_bf16_map_scan_is_as_accurate_as_the_walk(decay):
    maps, parts, S0 = _chunks(decay)
    ref = chunked.scan_start_states(maps, S0)          # f64
    scan, walk = _err(_scan_bf16(maps, S0), ref), _err(_walk_bf16(parts, S0), ref)
    # measured: scan 5.1e-3 / 2.9e-3 / 7.6e-5, walk 3.0e-3 / 3.4e-3 / 5.1e-3
    assert scan < 1e-2 and walk < 1e-2
    assert scan < 2.0 * walk, (scan, walk)
