"""Chunked restatement of the KDA variant (one decay gate per key channel) in f64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The KDA page ("KDA attention arm: per-group gradient proof on CUDA -- work log") names
the module's decay parameters and a chunked WY routine but prints neither the
recurrence nor the chunk algebra.  The recurrence the token oracle
(``gdn_oracle_kda_*``) states is the scalar-gate one with diag(g_t) in place of g_t:

    S_d = diag(g_t) S_{t-1},  delta_t = b_t (v_t - S_d^T k_t),  S_t = S_d + k_t delta_t^T,
    o_t = scale S_t^T q_t.

This module derives its chunked form, so that the algebra a chunked (tensor-core) kernel
would use is checked in f64 against the token oracle (``tests/test_oracle_chunked_kda.py``).
It is pinned against that oracle, never used to pin it.

Notation, per chunk of c tokens of one value head, rows r, s = 0..c-1, channels i:
  l = log g [c, Dk],  G = inclusive cumsum of l over the rows [c, Dk],
  M[r, s, i] = exp(G[r, i] - G[s, i]) for s <= r (every exponent <= 0),
  K, Q normalised keys / queries [c, Dk], V [c, Dv], b = beta [c], S chunk-start state.

Forward (an exact rewrite of the token recurrence):
  A[r, s] = b[r] sum_i K[r, i] K[s, i] M[r, s, i]   (s < r);   T = (I + A)^-1
  Kg = K * e^G,  Qg = Q * e^G       (row r decayed from the chunk start: exponents <= 0)
  U = T diag(b) V,  W = T diag(b) Kg,  Delta = U - W S
  P[r, s] = sum_i Q[r, i] K[s, i] M[r, s, i]   (s <= r)
  O = scale (Qg S + P Delta)
  S_next = diag(e^{G[c-1]}) S + (K * e^{G[c-1] - G})^T Delta

Unlike the scalar gate, M does not factor into one row factor times one column factor
that are both bounded: K * e^G times (K * e^{-G})^T does, but e^{-G} overflows once a
chunk decays by more than the float range.  ``gram`` therefore forms the two masked
products by blocks of ``sub`` rows.  A block of rows a against an earlier block of
columns is one plain product (X * e^{G - G[a0]}) (K * e^{G[a0] - G})^T, a0 being the
first row of block a, so both factors have exponents <= 0 (G does not increase along
the rows).  A block against itself is summed pair by pair over the channels.  With
``sub=None`` the whole chunk is summed pair by pair (the definition).

Backward: the reverse-mode derivative of each line above, in reverse order.
"""
from __future__ import annotations

import numpy as np

from .chunked import _l2, sigmoid, softplus


def gram(X, K, G, *, strict, sub=None):
    """sum_i X[r, i] K[s, i] exp(G[r, i] - G[s, i]) for s < r (strict) or s <= r, else 0."""
    c = X.shape[0]
    out = np.zeros((c, c))
    if sub is None:
        sub = c
    for a0 in range(0, c, sub):
        a1 = min(a0 + sub, c)
        # the block against itself, pair by pair
        for r in range(a0, a1):
            for s in range(a0, r + (0 if strict else 1)):
                out[r, s] = (X[r] * K[s] * np.exp(G[r] - G[s])).sum()
        # the block against every earlier column, through its first row
        if a0 > 0:
            Xr = X[a0:a1] * np.exp(G[a0:a1] - G[a0])
            Kc = K[:a0] * np.exp(G[a0] - G[:a0])
            out[a0:a1, :a0] = Xr @ Kc.T
    return out


def chunk_forward(Q, K, V, b, G, S, scale, sub=None):
    """One chunk forward.  G: [c, Dk] inclusive cumulative log-gates.  Returns
    (O, S_next, cache)."""
    c = Q.shape[0]
    A = b[:, None] * gram(K, K, G, strict=True, sub=sub)
    T = np.linalg.solve(np.eye(c) + A, np.eye(c))
    eG = np.exp(G)
    Kg, Qg = K * eG, Q * eG
    Bv, Bk = b[:, None] * V, b[:, None] * Kg
    U, W = T @ Bv, T @ Bk
    Delta = U - W @ S
    P = gram(Q, K, G, strict=False, sub=sub)
    O = scale * (Qg @ S + P @ Delta)
    eL = np.exp(G[-1])
    Kd = K * np.exp(G[-1] - G)
    S_next = eL[:, None] * S + Kd.T @ Delta
    cache = dict(A=A, T=T, eG=eG, Kg=Kg, Qg=Qg, Bv=Bv, Bk=Bk, W=W, Delta=Delta, P=P, eL=eL,
                 Kd=Kd)
    return O, S_next, cache


def _pair_terms(dX, X, K, G, strict):
    """Adjoint of Y[r, s] = sum_i X[r, i] K[s, i] exp(G[r, i] - G[s, i]) (masked) given
    dY: returns (dX, dK, dG), pair by pair."""
    c = X.shape[0]
    gX, gK, gG = np.zeros_like(X), np.zeros_like(K), np.zeros_like(G)
    for r in range(c):
        for s in range(r if strict else r + 1):
            if dX[r, s] == 0.0:
                continue
            m = np.exp(G[r] - G[s])
            gX[r] += dX[r, s] * K[s] * m
            gK[s] += dX[r, s] * X[r] * m
            t = dX[r, s] * X[r] * K[s] * m          # d/dG[r] of the term; -t for G[s]
            gG[r] += t
            gG[s] -= t
    return gX, gK, gG


def chunk_backward(Q, K, V, b, G, S, scale, dO, dS, cache):
    """Adjoint of :func:`chunk_forward` given dO and dS = dL/dS_next.
    Returns (dQ, dK, dV, db, dG, dS_prev); dG is [c, Dk]."""
    T, eG, Kg, Qg = cache["T"], cache["eG"], cache["Kg"], cache["Qg"]
    Bv, Bk, W, Delta, P = cache["Bv"], cache["Bk"], cache["W"], cache["Delta"], cache["P"]
    eL, Kd = cache["eL"], cache["Kd"]
    dG = np.zeros_like(G)
    # S_next = diag(eL) S + Kd^T Delta,  Kd = K * exp(G_last - G)
    dS_prev = eL[:, None] * dS
    dG[-1] += eL * (S * dS).sum(1)
    dKd = Delta @ dS.T
    dDelta = Kd @ dS
    dK = dKd * np.exp(G[-1] - G)
    X = dKd * Kd
    dG[-1] += X.sum(0)
    dG -= X
    # O = scale (Qg S + P Delta)
    dQg = scale * (dO @ S.T)
    dS_prev += scale * (Qg.T @ dO)
    dP = np.tril(scale * (dO @ Delta.T))
    dDelta += scale * (P.T @ dO)
    dQ = dQg * eG
    dG += dQg * Qg
    gQ, gK, gG = _pair_terms(dP, Q, K, G, strict=False)
    dQ += gQ
    dK += gK
    dG += gG
    # Delta = U - W S
    dU, dW = dDelta, -dDelta @ S.T
    dS_prev -= W.T @ dDelta
    # U = T Bv, W = T Bk, Bv = diag(b) V, Bk = diag(b) Kg, Kg = K * e^G
    dT = dU @ Bv.T + dW @ Bk.T
    dBv, dBk = T.T @ dU, T.T @ dW
    dV = b[:, None] * dBv
    db = (dBv * V).sum(1) + (dBk * Kg).sum(1)
    dKg = b[:, None] * dBk
    dK += dKg * eG
    dG += dKg * Kg
    # T = (I + A)^-1;  A[r, s] = b[r] sum_i K[r, i] K[s, i] M[r, s, i], s < r
    dA = np.tril(-(T.T @ dT @ T.T), -1)
    KKM = gram(K, K, G, strict=True)
    db += (dA * KKM).sum(1)
    gK1, gK2, gG = _pair_terms(b[:, None] * dA, K, K, G, strict=True)
    dK += gK1 + gK2
    dG += gG
    return dQ, dK, dV, db, dG, dS_prev


def _gates(alpha_h, beta_raw_h, a_log_h, b_alpha_h):
    """alpha_h [c, Dk], beta_raw_h [c], a_log_h scalar, b_alpha_h [Dk]."""
    b = sigmoid(beta_raw_h)
    x = alpha_h + b_alpha_h[None, :]
    l = -np.exp(a_log_h) * softplus(x)
    return b, x, l


def _key_head(h, Hk, r, head_map):
    return h % Hk if head_map else h // r


def forward(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, S0=None, *, Hk, Hv, Dk, Dv,
            scale=None, chunk=64, sub=None, head_map=0):
    """Chunked f64 forward over a varlen batch; the contract of ``oracle.kda_forward``
    (alpha [T, Hv*Dk], b_alpha [Hv*Dk])."""
    q, k, v, alpha = (np.asarray(x, np.float64) for x in (q, k, v, alpha))
    beta_raw, a_log = np.asarray(beta_raw, np.float64), np.asarray(a_log, np.float64)
    b_alpha = np.asarray(b_alpha, np.float64)
    scale = scale or 1.0 / np.sqrt(Dk)
    r = Hv // Hk
    cu = np.asarray(cu_seqlens, np.int64)
    N, Tt = len(cu) - 1, int(cu[-1])
    o = np.zeros((Tt, Hv * Dv))
    S_T = np.zeros((N, Hv, Dk, Dv))
    for n in range(N):
        for h in range(Hv):
            kh = _key_head(h, Hk, r, head_map)
            sk, sv, sa = (slice(kh * Dk, (kh + 1) * Dk), slice(h * Dv, (h + 1) * Dv),
                          slice(h * Dk, (h + 1) * Dk))
            S = np.zeros((Dk, Dv)) if S0 is None else np.array(S0[n, h], np.float64)
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                Q, _ = _l2(q[t0:t1, sk])
                K, _ = _l2(k[t0:t1, sk])
                b, _, l = _gates(alpha[t0:t1, sa], beta_raw[t0:t1, h], a_log[h], b_alpha[sa])
                O, S, _ = chunk_forward(Q, K, v[t0:t1, sv], b, np.cumsum(l, 0), S, scale, sub)
                o[t0:t1, sv] = O
            S_T[n, h] = S
    return o, S_T


def backward(q, k, v, alpha, beta_raw, a_log, b_alpha, cu_seqlens, dO, S0=None, dS_T=None, *,
             Hk, Hv, Dk, Dv, scale=None, chunk=64, head_map=0):
    """Chunked f64 backward; the contract of ``oracle.kda_backward``."""
    q, k, v, alpha, dO = (np.asarray(x, np.float64) for x in (q, k, v, alpha, dO))
    beta_raw, a_log = np.asarray(beta_raw, np.float64), np.asarray(a_log, np.float64)
    b_alpha = np.asarray(b_alpha, np.float64)
    scale = scale or 1.0 / np.sqrt(Dk)
    r = Hv // Hk
    cu = np.asarray(cu_seqlens, np.int64)
    N, Tt = len(cu) - 1, int(cu[-1])
    out = dict(dq=np.zeros((Tt, Hk * Dk)), dk=np.zeros((Tt, Hk * Dk)), dv=np.zeros((Tt, Hv * Dv)),
               dalpha=np.zeros((Tt, Hv * Dk)), dbeta_raw=np.zeros((Tt, Hv)), da_log=np.zeros(Hv),
               db_alpha=np.zeros(Hv * Dk), dS0=np.zeros((N, Hv, Dk, Dv)))
    for n in range(N):
        starts = list(range(int(cu[n]), int(cu[n + 1]), chunk))
        for h in range(Hv):
            kh = _key_head(h, Hk, r, head_map)
            sk, sv, sa = (slice(kh * Dk, (kh + 1) * Dk), slice(h * Dv, (h + 1) * Dv),
                          slice(h * Dk, (h + 1) * Dk))

            def chunk_inputs(t0):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                Q, nq = _l2(q[t0:t1, sk])
                K, nk = _l2(k[t0:t1, sk])
                b, x, l = _gates(alpha[t0:t1, sa], beta_raw[t0:t1, h], a_log[h], b_alpha[sa])
                return t1, Q, nq, K, nk, b, x, l

            S = np.zeros((Dk, Dv)) if S0 is None else np.array(S0[n, h], np.float64)
            states = []
            for t0 in starts:
                t1, Q, _, K, _, b, _, l = chunk_inputs(t0)
                states.append(S)
                _, S, _ = chunk_forward(Q, K, v[t0:t1, sv], b, np.cumsum(l, 0), S, scale)
            dS = np.zeros((Dk, Dv)) if dS_T is None else np.array(dS_T[n, h], np.float64)
            for ci in reversed(range(len(starts))):
                t0 = starts[ci]
                t1, Q, nq, K, nk, b, x, l = chunk_inputs(t0)
                V, G = v[t0:t1, sv], np.cumsum(l, 0)
                _, _, cache = chunk_forward(Q, K, V, b, G, states[ci], scale)
                dQ, dK, dV, db, dG, dS = chunk_backward(Q, K, V, b, G, states[ci], scale,
                                                        dO[t0:t1, sv], dS, cache)
                dl = np.cumsum(dG[::-1], 0)[::-1]       # l feeds every G at or after it
                dx = dl * (-np.exp(a_log[h])) * sigmoid(x)
                out["dv"][t0:t1, sv] = dV
                out["dalpha"][t0:t1, sa] = dx
                out["dbeta_raw"][t0:t1, h] = db * b * (1.0 - b)
                out["da_log"][h] += (dl * l).sum()
                out["db_alpha"][sa] += dx.sum(0)
                out["dq"][t0:t1, sk] += (dQ - Q * (dQ * Q).sum(1, keepdims=True)) / nq
                out["dk"][t0:t1, sk] += (dK - K * (dK * K).sum(1, keepdims=True)) / nk
            out["dS0"][n, h] = dS
    return out
