"""The chunked restatement of the KDA variant (oracle/chunked_kda.py) against the
token-by-token KDA oracle, in f64:

* forward and backward agree with the token oracle for chunks of 1, 16 and 64 tokens,
  ragged and empty sequences, both head maps, and Gram products formed whole or by
  blocks of 4 and 16 rows;
* with gates that differ strongly between channels (some channels lose 12 nats a token,
  others 0.01), a 64-token chunk decays by more than the f64 range: the single-factor
  product (K e^G)(K e^-G)^T overflows, while the blocked Gram product stays finite and
  agrees with the pairwise definition and with the token oracle;
* with the same gate on every channel of a head it equals the scalar-gate chunked
  restatement (oracle/chunked.py), which is pinned on its own;
* a design check for a tensor-core kernel: computed in fp32 with bf16 operands in every
  product, the blocked form stays within 1e-2 (about 5e-3 measured) of the token oracle,
  inside the 2e-2 bar of bf16 outputs;
* the same with a block's own pairs also formed as a bf16 product through the block's
  first row, wherever the block decays by at most e^60 (the kernel's choice), for gates
  whose blocks sit just below and just above that bound.
"""
import numpy as np
import pytest

import oracle
from oracle import chunked, chunked_kda


def _inputs(seed, seqlens=(37, 0, 70), Hk=2, Hv=4, Dk=8, Dv=6, strong=False):
    rng = np.random.default_rng(seed)
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    d = dict(q=rng.standard_normal((T, Hk * Dk)), k=rng.standard_normal((T, Hk * Dk)),
             v=rng.standard_normal((T, Hv * Dv)), alpha=rng.standard_normal((T, Hv * Dk)),
             beta_raw=rng.standard_normal((T, Hv)), a_log=0.5 * rng.standard_normal(Hv),
             b_alpha=0.3 * rng.standard_normal(Hv * Dk),
             S0=0.5 * rng.standard_normal((len(seqlens), Hv, Dk, Dv)),
             dO=rng.standard_normal((T, Hv * Dv)),
             dS_T=rng.standard_normal((len(seqlens), Hv, Dk, Dv)))
    if strong:
        # even channels: softplus(12) ~ 12 nats a token; odd channels: ~0.01
        d["a_log"][:] = 0.0
        d["b_alpha"][:] = 0.0
        x = d["alpha"].reshape(T, Hv, Dk)
        x[:, :, 0::2] = 12.0 + 0.1 * x[:, :, 0::2]
        x[:, :, 1::2] = np.log(np.expm1(0.01)) + 0.1 * x[:, :, 1::2]
    return d, cu, dict(Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)


def _rel(a, b):
    den = np.abs(b).max()
    return np.abs(a - b).max() / (den if den > 0 else 1.0)


def _token_fwd(d, cu, kw, head_map=0):
    return oracle.kda_forward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                              d["b_alpha"], cu, d["S0"], head_map=head_map, **kw)


def _token_bwd(d, cu, kw, head_map=0):
    return oracle.kda_backward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                               d["b_alpha"], cu, d["dO"], d["S0"], d["dS_T"], head_map=head_map,
                               **kw)


@pytest.mark.parametrize("chunk,sub", [(1, None), (16, None), (16, 4), (64, None), (64, 16)])
@pytest.mark.parametrize("head_map", [0, 1])
def test_chunked_forward_equals_token_oracle(chunk, sub, head_map):
    d, cu, kw = _inputs(1)
    o, S_T = _token_fwd(d, cu, kw, head_map)
    oc, Sc = chunked_kda.forward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                                 d["b_alpha"], cu, d["S0"], chunk=chunk, sub=sub,
                                 head_map=head_map, **kw)
    assert _rel(oc, o) < 1e-12 and _rel(Sc, S_T) < 1e-12


@pytest.mark.parametrize("chunk,head_map", [(16, 0), (64, 0), (64, 1)])
def test_chunked_backward_equals_token_oracle(chunk, head_map):
    d, cu, kw = _inputs(2, seqlens=(21, 0, 40))
    g = _token_bwd(d, cu, kw, head_map)
    gc = chunked_kda.backward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                              d["b_alpha"], cu, d["dO"], d["S0"], d["dS_T"], chunk=chunk,
                              head_map=head_map, **kw)
    for key in g:
        assert gc[key].shape == g[key].shape, key
        assert _rel(gc[key], g[key]) < 1e-11, (key, _rel(gc[key], g[key]))


def test_blocked_gram_stays_finite_where_one_factor_overflows():
    d, cu, kw = _inputs(3, seqlens=(64,), Hk=1, Hv=1, strong=True)
    Dk = kw["Dk"]
    K, _ = chunked._l2(d["k"][:, :Dk])
    b, _, l = chunked_kda._gates(d["alpha"][:, :Dk], d["beta_raw"][:, 0], d["a_log"][0],
                                 d["b_alpha"][:Dk])
    G = np.cumsum(l, 0)
    assert -G.min() > 709.0                         # e^-G leaves the f64 range
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.tril((K * np.exp(G)) @ (K * np.exp(-G)).T, -1)
    assert not np.isfinite(naive).all()
    pair = chunked_kda.gram(K, K, G, strict=True)
    blocked = chunked_kda.gram(K, K, G, strict=True, sub=16)
    assert np.isfinite(blocked).all()
    assert _rel(blocked, pair) < 1e-14
    o, S_T = _token_fwd(d, cu, kw)
    oc, Sc = chunked_kda.forward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                                 d["b_alpha"], cu, d["S0"], chunk=64, sub=16, **kw)
    assert _rel(oc, o) < 1e-12 and _rel(Sc, S_T) < 1e-12


def test_equal_channel_gates_equal_the_scalar_chunked_form():
    d, cu, kw = _inputs(4, seqlens=(50, 13))
    Hv, Dk = kw["Hv"], kw["Dk"]
    rng = np.random.default_rng(9)
    a_s = rng.standard_normal((int(cu[-1]), Hv))
    dt = 0.3 * rng.standard_normal(Hv)
    d["alpha"], d["b_alpha"] = np.repeat(a_s, Dk, axis=1), np.repeat(dt, Dk)
    oc, Sc = chunked_kda.forward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                                 d["b_alpha"], cu, d["S0"], chunk=16, sub=4, **kw)
    o, S = chunked.forward(d["q"], d["k"], d["v"], a_s, d["beta_raw"], d["a_log"], dt, cu,
                           d["S0"], chunk=16, **kw)
    assert _rel(oc, o) < 1e-12 and _rel(Sc, S) < 1e-12


def _bf16(x):
    """Round to bfloat16 (nearest even), returned as float32."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def _blocked_forward_bf16_operands(d, cu, kw, chunk=64, sub=16, diag_product=False,
                                   wide=60.0, stats=None):
    """The blocked chunked forward with the arithmetic a tensor-core kernel would use: fp32
    throughout, and every product (the off-diagonal Gram blocks, U, W, W S, Qg S, P Delta
    and the state update) fed bf16-rounded operands with fp32 accumulation.  The
    triangular solve stays fp32.  The diagonal Gram blocks are fp32 pairwise sums, or,
    with diag_product, products of bf16 operands through the block's first row as well
    (X e^{G - G[a0]} against K e^{G[a0] - G}, masked to the lower triangle) wherever the
    block's own decay (the sum of its rows' log gates) stays below `wide` on every
    channel; `stats` (a list) then collects each such block's decay."""
    f = lambda a: np.asarray(a, np.float32)

    def gram(X, K, G, strict):
        c = X.shape[0]
        out = np.zeros((c, c), np.float32)
        for a0 in range(0, c, sub):
            a1 = min(a0 + sub, c)
            decay = float(((G[a0 - 1] if a0 > 0 else 0.0) - G[a1 - 1]).max())
            if diag_product and decay <= wide:
                full = _bf16(X[a0:a1] * np.exp(G[a0:a1] - G[a0])) @ \
                    _bf16(K[a0:a1] * np.exp(G[a0] - G[a0:a1])).T
                assert np.isfinite(full).all()   # the masked entries above the diagonal too
                out[a0:a1, a0:a1] = np.tril(full, -1 if strict else 0)
                if stats is not None:
                    stats.append(decay)
            else:
                for r in range(a0, a1):
                    for s in range(a0, r + (0 if strict else 1)):
                        out[r, s] = (X[r] * K[s] * np.exp(G[r] - G[s])).sum(dtype=np.float32)
            if a0 > 0:
                out[a0:a1, :a0] = _bf16(X[a0:a1] * np.exp(G[a0:a1] - G[a0])) @ \
                    _bf16(K[:a0] * np.exp(G[a0] - G[:a0])).T
        return out

    Hk, Hv, Dk, Dv = kw["Hk"], kw["Hv"], kw["Dk"], kw["Dv"]
    scale = np.float32(1.0 / np.sqrt(Dk))
    r = Hv // Hk
    o = np.zeros((int(cu[-1]), Hv * Dv), np.float32)
    S_T = np.zeros((len(cu) - 1, Hv, Dk, Dv), np.float32)
    for n in range(len(cu) - 1):
        for h in range(Hv):
            sk = slice((h // r) * Dk, (h // r + 1) * Dk)
            sv, sa = slice(h * Dv, (h + 1) * Dv), slice(h * Dk, (h + 1) * Dk)
            S = f(d["S0"][n, h])
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                Q, K = (f(chunked._l2(d[x][t0:t1, sk])[0]) for x in ("q", "k"))
                b, _, l = chunked_kda._gates(d["alpha"][t0:t1, sa], d["beta_raw"][t0:t1, h],
                                             d["a_log"][h], d["b_alpha"][sa])
                b, G, V = f(b), f(np.cumsum(l, 0)), f(d["v"][t0:t1, sv])
                c = t1 - t0
                A = b[:, None] * gram(K, K, G, True)
                T = f(np.linalg.solve(np.eye(c) + A, np.eye(c)))
                eG = np.exp(G)
                U = _bf16(T) @ _bf16(b[:, None] * V)
                W = _bf16(T) @ _bf16(b[:, None] * K * eG)
                Delta = U - _bf16(W) @ _bf16(S)
                P = gram(Q, K, G, False)
                o[t0:t1, sv] = scale * (_bf16(Q * eG) @ _bf16(S) + _bf16(P) @ _bf16(Delta))
                S = np.exp(G[-1])[:, None] * S + _bf16(K * np.exp(G[-1] - G)).T @ _bf16(Delta)
            S_T[n, h] = S
    return o, S_T


@pytest.mark.parametrize("strong", [False, True])
def test_blocked_form_with_bf16_operands_stays_inside_the_bf16_bar(strong):
    """Design check for a tensor-core chunked KDA: the blocked form, computed in fp32 with
    bf16 operands in every product, stays well inside the bf16 bar (2e-2 of max|ref|) of
    the f64 token oracle, for typical gates and for gates that decay 12 nats a token on
    half the channels."""
    d, cu, kw = _inputs(11, seqlens=(150, 41), Hk=1, Hv=2, Dk=32, Dv=32, strong=strong)
    o, S_T = _token_fwd(d, cu, kw)
    oc, Sc = _blocked_forward_bf16_operands(d, cu, kw)
    assert np.isfinite(oc).all() and np.isfinite(Sc).all()
    assert _rel(oc, o) < 1e-2 and _rel(Sc, S_T) < 1e-2


@pytest.mark.parametrize("gates", ["typical", "near_e60", "strong"])
def test_diagonal_blocks_through_the_product_stay_inside_the_bf16_bar(gates):
    """Design check of the tensor-core kernel's own choice: a 16-row block's own pairs also
    go through the bf16 product, referenced to the block's first row, wherever the block
    decays by at most e^60 on every channel (the operand factor K e^{G[a0] - G} then
    reaches e^60, and the masked entries above the diagonal stay finite in fp32); faster
    blocks keep the pairwise sums.  With typical gates, with half the channels losing
    ~3.7 nats a token (blocks just below and above e^60) and with 12 nats a token, the
    forward stays inside the bf16 bar of the f64 token oracle."""
    d, cu, kw = _inputs(13, seqlens=(150, 41), Hk=1, Hv=2, Dk=32, Dv=32,
                        strong=gates == "strong")
    if gates == "near_e60":
        rng = np.random.default_rng(5)
        d["a_log"][:] = 0.0
        d["b_alpha"][:] = 0.0
        x = d["alpha"].reshape(int(cu[-1]), kw["Hv"], kw["Dk"])
        x[:, :, 0::2] = 3.7 + 0.05 * rng.standard_normal(x[:, :, 0::2].shape)
    o, S_T = _token_fwd(d, cu, kw)
    stats = []
    oc, Sc = _blocked_forward_bf16_operands(d, cu, kw, diag_product=True, stats=stats)
    assert np.isfinite(oc).all() and np.isfinite(Sc).all()
    assert _rel(oc, o) < 1e-2 and _rel(Sc, S_T) < 1e-2
    if gates == "typical":
        assert stats and max(stats) < 60.0
    if gates == "near_e60":
        assert stats and max(stats) > 55.0     # factors near e^60 were exercised
    if gates == "strong":
        assert not stats                       # every block decays past e^60

