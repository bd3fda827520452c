"""Pins of the oracle's KDA variant (a decay gate per key channel) to facts other than its
own code:

* with the same alpha and b_alpha on every channel of a head it is the scalar-gate
  recurrence, whose oracle is pinned on its own: the same o, S_T, dq, dk, dv, dbeta_raw,
  dS_0 and d a_log, and the channel sums of dalpha / d b_alpha equal dalpha / d dt_bias;
* central differences (f64) of the forward pin every gradient;
* a channel that no key touches only decays: row c of S_T is (prod_t g_t[c]) S_0[c].
A gate applied to the wrong axis (value instead of key channels), after the retrieval
instead of before, or a dropped channel in dg fails one of them.
"""
import numpy as np
import pytest

import oracle


def _inputs(seed, T=(4, 3), Hk=1, Hv=2, Dk=4, Dv=3):
    rng = np.random.default_rng(seed)
    Tt = sum(T)
    cu = np.concatenate([[0], np.cumsum(T)]).astype(np.int32)
    d = dict(q=rng.standard_normal((Tt, Hk * Dk)), k=rng.standard_normal((Tt, Hk * Dk)),
             v=rng.standard_normal((Tt, Hv * Dv)), alpha=rng.standard_normal((Tt, Hv * Dk)),
             beta_raw=rng.standard_normal((Tt, Hv)), a_log=0.5 * rng.standard_normal(Hv),
             b_alpha=0.3 * rng.standard_normal(Hv * Dk),
             S0=0.5 * rng.standard_normal((len(T), Hv, Dk, Dv)),
             dO=rng.standard_normal((Tt, Hv * Dv)),
             dS_T=rng.standard_normal((len(T), Hv, Dk, Dv)))
    return d, cu, dict(Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)


def _fwd(d, cu, kw):
    return oracle.kda_forward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                              d["b_alpha"], cu, d["S0"], **kw)


def _bwd(d, cu, kw):
    return oracle.kda_backward(d["q"], d["k"], d["v"], d["alpha"], d["beta_raw"], d["a_log"],
                               d["b_alpha"], cu, d["dO"], d["S0"], d["dS_T"], **kw)


@pytest.mark.parametrize("Hk,Hv", [(1, 2), (2, 4)])
def test_equal_channel_gates_reduce_to_the_scalar_gate(Hk, Hv):
    d, cu, kw = _inputs(1, Hk=Hk, Hv=Hv)
    Dk = kw["Dk"]
    rng = np.random.default_rng(2)
    a_s = rng.standard_normal((cu[-1], Hv))
    dt = 0.3 * rng.standard_normal(Hv)
    d["alpha"] = np.repeat(a_s, Dk, axis=1)          # column h*Dk + c = a_s[:, h]
    d["b_alpha"] = np.repeat(dt, Dk)
    o, S_T = _fwd(d, cu, kw)
    o_r, S_r = oracle.forward(d["q"], d["k"], d["v"], a_s, d["beta_raw"], d["a_log"], dt, cu,
                              d["S0"], **kw)
    assert np.allclose(o, o_r, rtol=0, atol=1e-12) and np.allclose(S_T, S_r, rtol=0, atol=1e-12)
    g = _bwd(d, cu, kw)
    r = oracle.backward(d["q"], d["k"], d["v"], a_s, d["beta_raw"], d["a_log"], dt, cu, d["dO"],
                        d["S0"], d["dS_T"], **kw)
    for key in ("dq", "dk", "dv", "dbeta_raw", "dS0", "da_log"):
        assert np.allclose(g[key], r[key], rtol=0, atol=1e-11), key
    T = cu[-1]
    assert np.allclose(g["dalpha"].reshape(T, Hv, Dk).sum(-1), r["dalpha"], rtol=0, atol=1e-11)
    assert np.allclose(g["db_alpha"].reshape(Hv, Dk).sum(-1), r["ddt_bias"], rtol=0, atol=1e-11)


def test_gradients_match_central_differences():
    d, cu, kw = _inputs(3)
    g = _bwd(d, cu, kw)

    def loss(dd):
        o, S_T = _fwd(dd, cu, kw)
        return float((o * d["dO"]).sum() + (S_T * d["dS_T"]).sum())

    names = {"q": "dq", "k": "dk", "v": "dv", "alpha": "dalpha", "beta_raw": "dbeta_raw",
             "a_log": "da_log", "b_alpha": "db_alpha", "S0": "dS0"}
    h = 1e-6
    for x, gx in names.items():
        fd = np.zeros_like(d[x])
        it = np.nditer(d[x], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            dp = {k: (v.copy() if k == x else v) for k, v in d.items()}
            dm = {k: (v.copy() if k == x else v) for k, v in d.items()}
            dp[x][i] += h
            dm[x][i] -= h
            fd[i] = (loss(dp) - loss(dm)) / (2 * h)
        err = np.abs(fd - g[gx]).max() / max(np.abs(g[gx]).max(), 1e-30)
        assert err < 2e-7, (x, err)


def test_untouched_channels_only_decay():
    d, cu, kw = _inputs(5, T=(6,))
    Dk, Hv = kw["Dk"], kw["Hv"]
    d["k"][:, 2:] = 0.0                               # keys live in channels 0 and 1
    _, S_T = _fwd(d, cu, kw)
    x = d["alpha"].reshape(-1, Hv, Dk) + d["b_alpha"].reshape(Hv, Dk)[None]
    ell = -np.exp(d["a_log"])[None, :, None] * np.logaddexp(0.0, x)    # [T, Hv, Dk]
    decay = np.exp(ell.sum(0))                                          # [Hv, Dk]
    for h in range(Hv):
        for c in (2, 3):
            assert np.allclose(S_T[0, h, c], decay[h, c] * d["S0"][0, h, c], rtol=1e-13, atol=0)
