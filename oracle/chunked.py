"""Chunked (WY / UT) restatement of the Gated DeltaNet recurrence in f64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages state the recurrence token by token (lattice-inference 0.6.0,
src/attention/gdn_backward.rs, module header "Forward recap" and
gdn_backward section 4).  They name a chunked form only by function name
(``chunk_wy_forward_impl`` and ``ChunkWy::backward`` on the "KDA attention
arm: per-group gradient proof on CUDA" work log) and never write it out.  This
module derives it from the token recurrence so that the algebra the CUDA path
uses can be checked, in f64, against the token-by-token oracle.  It is pinned
against that oracle (``tests/test_oracle_pins.py``), never used to pin it.

Notation, per chunk of c <= C tokens of one value head, rows r, s = 0..c-1:
  l = log g,  G = inclusive cumsum(l),  E[r, s] = exp(G[r] - G[s]) for s <= r,
  K, Q = L2-normalised keys / queries [c, Dk], V [c, Dv], b = beta [c],
  S = state at the chunk start [Dk, Dv].

Forward (exact rewrite of the token recurrence):
  A = diag(b) (E * K K^T), strictly lower;  T = (I + A)^-1
  U = T diag(b) V;  W = T diag(b * e^G) K;  Delta = U - W S
  P = E * (Q K^T), lower incl. diagonal
  O = scale (diag(e^G) Q S + P Delta)
  S_next = e^{G[c-1]} S + K^T diag(e^{G[c-1] - G}) Delta

Backward: reverse-mode derivative of each line above, in reverse order.
"""
from __future__ import annotations

import numpy as np


def softplus(x):
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _l2(x):
    n = np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)
    return x / n, n


def _decay_matrix(G):
    c = G.shape[0]
    low = np.tril(np.ones((c, c), dtype=bool))
    diff = np.where(low, G[:, None] - G[None, :], 0.0)
    return np.where(low, np.exp(diff), 0.0), low


def chunk_forward(Q, K, V, b, G, S, scale):
    """One chunk forward.  Returns (O, S_next, cache)."""
    c = Q.shape[0]
    E, low = _decay_matrix(G)
    strict = np.tril(np.ones((c, c), dtype=bool), -1)
    A = np.where(strict, b[:, None] * E * (K @ K.T), 0.0)
    T = np.linalg.solve(np.eye(c) + A, np.eye(c))
    Bv = b[:, None] * V
    Bk = (b * np.exp(G))[:, None] * K
    U = T @ Bv
    W = T @ Bk
    Delta = U - W @ S
    P = np.where(low, E * (Q @ K.T), 0.0)
    eG = np.exp(G)
    O = scale * (eG[:, None] * (Q @ S) + P @ Delta)
    cdec = np.exp(G[-1] - G)
    S_next = np.exp(G[-1]) * S + K.T @ (cdec[:, None] * Delta)
    cache = dict(E=E, low=low, strict=strict, A=A, T=T, Bv=Bv, Bk=Bk, W=W, U=U, Delta=Delta,
                 P=P, eG=eG, cdec=cdec)
    return O, S_next, cache


def chunk_backward(Q, K, V, b, G, S, scale, dO, dS, cache):
    """Adjoint of :func:`chunk_forward` given dO and dS = dL/dS_next.
    Returns (dQ, dK, dV, db, dG, dS_prev)."""
    E, low, strict = cache["E"], cache["low"], cache["strict"]
    A, T, Bv, Bk, W = cache["A"], cache["T"], cache["Bv"], cache["Bk"], cache["W"]
    Delta, P, eG, cdec = cache["Delta"], cache["P"], cache["eG"], cache["cdec"]
    c = Q.shape[0]
    dG = np.zeros(c)
    # S_next = e^{G_last} S + K^T diag(cdec) Delta
    dDelta = scale * (P.T @ dO) + cdec[:, None] * (K @ dS)
    dS_prev = np.exp(G[-1]) * dS + scale * (Q.T @ (eG[:, None] * dO))
    dK = cdec[:, None] * (Delta @ dS.T)
    dcdec = ((K @ dS) * Delta).sum(1)
    dG[-1] += np.exp(G[-1]) * (S * dS).sum() + (dcdec * cdec).sum()
    dG -= dcdec * cdec
    # O = scale (diag(e^G) Q S + P Delta)
    dP = np.where(low, scale * (dO @ Delta.T), 0.0)
    dQ = scale * eG[:, None] * (dO @ S.T) + (dP * E) @ K
    dK += (dP * E).T @ Q
    dG += scale * eG * (dO * (Q @ S)).sum(1)
    X = dP * P
    dG += X.sum(1) - X.sum(0)
    # Delta = U - W S
    dU = dDelta
    dW = -dDelta @ S.T
    dS_prev -= W.T @ dDelta
    # U = T Bv, W = T Bk
    dT = dU @ Bv.T + dW @ Bk.T
    dBv = T.T @ dU
    dBk = T.T @ dW
    dV = b[:, None] * dBv
    db = (dBv * V).sum(1)
    dK += (b * eG)[:, None] * dBk
    t = (dBk * K).sum(1)
    db += eG * t
    dG += b * eG * t
    # T = (I + A)^-1, A strictly lower
    dA = np.where(strict, -(T.T @ dT @ T.T), 0.0)
    KK = K @ K.T
    db += (dA * E * KK).sum(1)
    Y = dA * A
    dG += Y.sum(1) - Y.sum(0)
    H = dA * b[:, None] * E
    dK += H @ K + H.T @ K
    return dQ, dK, dV, db, dG, dS_prev


def _gates(alpha, beta_raw, a_log, dt_bias):
    b = sigmoid(beta_raw)
    x = alpha + dt_bias
    l = -np.exp(a_log) * softplus(x)
    return b, x, l


def forward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, S0=None, *, Hk, Hv, Dk, Dv,
            scale=None, chunk=64):
    """Chunked f64 forward over a varlen batch.  Same contract as ``oracle.forward``."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta_raw = np.asarray(alpha, np.float64), np.asarray(beta_raw, np.float64)
    a_log, dt_bias = np.asarray(a_log, np.float64), np.asarray(dt_bias, np.float64)
    scale = scale or 1.0 / np.sqrt(Dk)
    r = Hv // Hk
    cu = np.asarray(cu_seqlens, np.int64)
    N, T = len(cu) - 1, int(cu[-1])
    o = np.zeros((T, Hv * Dv))
    S_T = np.zeros((N, Hv, Dk, Dv))
    for n in range(N):
        for h in range(Hv):
            kh = h // r
            S = np.zeros((Dk, Dv)) if S0 is None else np.array(S0[n, h], np.float64)
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                Q, _ = _l2(q[t0:t1, kh * Dk:(kh + 1) * Dk])
                K, _ = _l2(k[t0:t1, kh * Dk:(kh + 1) * Dk])
                V = v[t0:t1, h * Dv:(h + 1) * Dv]
                b, _, l = _gates(alpha[t0:t1, h], beta_raw[t0:t1, h], a_log[h], dt_bias[h])
                O, S, _ = chunk_forward(Q, K, V, b, np.cumsum(l), S, scale)
                o[t0:t1, h * Dv:(h + 1) * Dv] = O
            S_T[n, h] = S
    return o, S_T


def backward(q, k, v, alpha, beta_raw, a_log, dt_bias, cu_seqlens, dO, S0=None, dS_T=None, *,
             Hk, Hv, Dk, Dv, scale=None, chunk=64):
    """Chunked f64 backward.  Same contract as ``oracle.backward``."""
    q, k, v, dO = (np.asarray(x, np.float64) for x in (q, k, v, dO))
    alpha, beta_raw = np.asarray(alpha, np.float64), np.asarray(beta_raw, np.float64)
    a_log, dt_bias = np.asarray(a_log, np.float64), np.asarray(dt_bias, np.float64)
    scale = scale or 1.0 / np.sqrt(Dk)
    r = Hv // Hk
    cu = np.asarray(cu_seqlens, np.int64)
    N, T = len(cu) - 1, int(cu[-1])
    out = dict(dq=np.zeros((T, Hk * Dk)), dk=np.zeros((T, Hk * Dk)), dv=np.zeros((T, Hv * Dv)),
               dalpha=np.zeros((T, Hv)), dbeta_raw=np.zeros((T, Hv)), da_log=np.zeros(Hv),
               ddt_bias=np.zeros(Hv), dS0=np.zeros((N, Hv, Dk, Dv)))
    for n in range(N):
        starts = list(range(int(cu[n]), int(cu[n + 1]), chunk))
        for h in range(Hv):
            kh = h // r
            sl_k = slice(kh * Dk, (kh + 1) * Dk)
            sl_v = slice(h * Dv, (h + 1) * Dv)
            # forward sweep: chunk-start states
            S = np.zeros((Dk, Dv)) if S0 is None else np.array(S0[n, h], np.float64)
            states = []
            for t0 in starts:
                t1 = min(t0 + chunk, int(cu[n + 1]))
                K, _ = _l2(k[t0:t1, sl_k])
                Q, _ = _l2(q[t0:t1, sl_k])
                b, _, l = _gates(alpha[t0:t1, h], beta_raw[t0:t1, h], a_log[h], dt_bias[h])
                states.append(S)
                _, S, _ = chunk_forward(Q, K, v[t0:t1, sl_v], b, np.cumsum(l), S, scale)
            dS = np.zeros((Dk, Dv)) if dS_T is None else np.array(dS_T[n, h], np.float64)
            for ci in reversed(range(len(starts))):
                t0 = starts[ci]
                t1 = min(t0 + chunk, int(cu[n + 1]))
                Q, nq = _l2(q[t0:t1, sl_k])
                K, nk = _l2(k[t0:t1, sl_k])
                V = v[t0:t1, sl_v]
                b, x, l = _gates(alpha[t0:t1, h], beta_raw[t0:t1, h], a_log[h], dt_bias[h])
                G = np.cumsum(l)
                _, _, cache = chunk_forward(Q, K, V, b, G, states[ci], scale)
                dQ, dK, dV, db, dG, dS = chunk_backward(Q, K, V, b, G, states[ci], scale,
                                                        dO[t0:t1, sl_v], dS, cache)
                dl = np.cumsum(dG[::-1])[::-1]          # l feeds every G at or after it
                dalpha = dl * (-np.exp(a_log[h])) * sigmoid(x)
                out["dv"][t0:t1, sl_v] = dV
                out["dalpha"][t0:t1, h] = dalpha
                out["dbeta_raw"][t0:t1, h] = db * b * (1.0 - b)
                out["da_log"][h] += (dl * l).sum()
                out["ddt_bias"][h] += dalpha.sum()
                out["dq"][t0:t1, sl_k] += (dQ - Q * (dQ * Q).sum(1, keepdims=True)) / nq
                out["dk"][t0:t1, sl_k] += (dK - K * (dK * K).sum(1, keepdims=True)) / nk
            out["dS0"][n, h] = dS
    return out


# ---------------------------------------------------------------------------
# Chunk maps.  A chunk maps its start state affinely to its end state,
#   S_next = Phi S + R,  Phi = e^{G[c-1]} I - (diag(cdec) K)^T W  (Dk x Dk),
#   R = (diag(cdec) K)^T U  (Dk x Dv),
# both from the chunk's own inputs (the last line of the forward above with
# Delta = U - W S expanded).  The reverse carry is affine with the transposed map:
#   dS_prev = Phi^T dS + Gc,  Gc = scale Q^T diag(e^G) dO - W^T (scale P^T dO).
# So the chunk-start states of a sequence are a prefix scan of the maps, which a
# log-depth scan forms in ceil(log2 n) rounds instead of n dependent chunk steps.

def chunk_map(Q, K, V, b, G, scale):
    """(Phi, R) of one chunk."""
    _, _, cache = chunk_forward(Q, K, V, b, G, np.zeros((K.shape[1], V.shape[1])), scale)
    Kd = cache["cdec"][:, None] * K
    Phi = np.exp(G[-1]) * np.eye(K.shape[1]) - Kd.T @ cache["W"]
    return Phi, Kd.T @ cache["U"]


def chunk_carry_term(Q, K, V, b, G, scale, dO):
    """Gc of one chunk: the start-state gradient when the end-state gradient is zero."""
    _, _, cache = chunk_forward(Q, K, V, b, G, np.zeros((K.shape[1], V.shape[1])), scale)
    return scale * (Q.T @ (cache["eG"][:, None] * dO)) - cache["W"].T @ (scale * (cache["P"].T @ dO))


def compose(later, earlier):
    """The map of `earlier` followed by `later`: (P2, R2) o (P1, R1) = (P2 P1, P2 R1 + R2)."""
    (P2, R2), (P1, R1) = later, earlier
    return P2 @ P1, P2 @ R1 + R2


def scan_start_states(maps, S0):
    """State at the start of every chunk from the chunk maps, by a log-depth inclusive
    scan (Hillis-Steele: in round j every prefix takes in the one 2^j chunks before it)."""
    pre = list(maps)
    step = 1
    while step < len(pre):
        pre = [pre[i] if i < step else compose(pre[i], pre[i - step]) for i in range(len(pre))]
        step *= 2
    return [S0] + [P @ S0 + R for P, R in pre[:-1]]
