"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Each test ties the f64 oracle to something the pages or the mathematics fix
independently of the oracle's own code:

* central finite differences of the oracle's forward pin every gradient of
  its backward (the gradcheck method of lattice-inference's gdn_backward.rs
  tests, run here in f64 end to end so no f32 noise floor arises);
* closed forms and invariants of the recurrence (the delta rule's write makes
  the state retrieve what was written; beta = 0 with g = 1 leaves the state
  untouched; beta = 0 decays it by exp(sum log g), with softplus taken from
  numpy's logaddexp);
* structural identities: heads are independent, a shared key head equals an
  explicit repeat with the q/k gradients summed, varlen packing equals separate
  runs, the state and output are linear in (v, S_0) for fixed gates and keys;
* zero upstream gradient gives exactly zero gradients;
* the chunked numpy restatement (the algebra the GPU path implements) agrees
  with the token-by-token oracle for chunk sizes 1, 16 and 64.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import chunked

FIELDS = ("q", "k", "v", "alpha", "beta_raw", "a_log", "dt_bias", "S0")


def _draw(Hk, Hv, Dk, Dv, seqlens, seed, S0=True, dST=True, dt=True):
    wl = W.custom(Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=seqlens, seed=seed, packed=True,
                  S0_std=0.5 if S0 else 0.0, dST_std=0.3 if dST else 0.0,
                  dt_bias_std=0.5 if dt else 0.0)
    inp = W.generate(wl)
    arrs = dict(q=np.array(inp.q, np.float64), k=np.array(inp.k, np.float64),
                v=np.array(inp.v, np.float64), alpha=inp.alpha.astype(np.float64),
                beta_raw=inp.beta_raw.astype(np.float64), a_log=inp.a_log.astype(np.float64),
                dt_bias=inp.dt_bias.astype(np.float64),
                S0=None if inp.S0 is None else inp.S0.astype(np.float64))
    return wl, inp, arrs


def _fwd(wl, cu, a, **kw):
    return oracle.forward(a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"], a["a_log"],
                          a["dt_bias"], cu, a["S0"], Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv,
                          n_threads=1, **kw)


def _bwd(wl, cu, a, dO, dS_T, **kw):
    return oracle.backward(a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"], a["a_log"],
                           a["dt_bias"], cu, dO, a["S0"], dS_T, Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk,
                           Dv=wl.Dv, n_threads=1, **kw)


def _rel(a, b):
    den = np.abs(b).max()
    return np.abs(a - b).max() / (den if den > 0 else 1.0)


FD_CASES = [
    # Hk, Hv, Dk, Dv, seqlens, seed, segment
    (1, 1, 4, 4, (1,), 11, 64),
    (1, 3, 4, 6, (5, 3), 12, 2),
    (2, 4, 8, 4, (20,), 13, 7),
    (2, 6, 4, 8, (6, 0, 9), 14, 4),
]


@pytest.mark.parametrize("case", FD_CASES, ids=lambda c: "Hk%d_Hv%d_Dk%d_Dv%d_T%s" % (
    c[0], c[1], c[2], c[3], "-".join(map(str, c[4]))))
def test_backward_matches_central_differences(case):
    Hk, Hv, Dk, Dv, seqlens, seed, segment = case
    wl, inp, a = _draw(Hk, Hv, Dk, Dv, seqlens, seed)
    cu = inp.cu_seqlens
    rng = np.random.default_rng(seed)
    dO = rng.standard_normal((wl.total_tokens, Hv * Dv))
    dS_T = rng.standard_normal((wl.n_seqs, Hv, Dk, Dv))

    def loss(arrs):
        o, S_T = _fwd(wl, cu, arrs)
        return float((o * dO).sum() + (S_T * dS_T).sum())

    g = _bwd(wl, cu, a, dO, dS_T, segment=segment)
    names = dict(q="dq", k="dk", v="dv", alpha="dalpha", beta_raw="dbeta_raw", a_log="da_log",
                 dt_bias="ddt_bias", S0="dS0")
    h = 1e-6
    for f in FIELDS:
        base = a[f]
        fd = np.zeros_like(base)
        flat, fdf = base.reshape(-1), fd.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(a)
            flat[i] = old - h
            lm = loss(a)
            flat[i] = old
            fdf[i] = (lp - lm) / (2 * h)
        an = g[names[f]]
        assert np.abs(an).max() > 0, f
        err = _rel(an.reshape(fd.shape), fd)
        assert err < 2e-7, (f, err)


def test_t1_closed_form_forward_and_backward():
    """One token from a nonzero S_0: S_1 = g S_0 + k (b (v - g S_0^T k))^T, o = scale S_1^T q,
    and the hand-derived gradients of L = <dO, o> + <dS_T, S_1>."""
    wl, inp, a = _draw(1, 1, 5, 3, (1,), 21)
    q = a["q"][0] / np.sqrt((a["q"][0] ** 2).sum() + 1e-6)
    k = a["k"][0] / np.sqrt((a["k"][0] ** 2).sum() + 1e-6)
    v = a["v"][0]
    S0 = a["S0"][0, 0]
    b = 1 / (1 + np.exp(-a["beta_raw"][0, 0]))
    g = np.exp(-np.exp(a["a_log"][0]) * np.logaddexp(0, a["alpha"][0, 0] + a["dt_bias"][0]))
    scale = 1 / np.sqrt(5)
    S1 = g * S0 + np.outer(k, b * (v - g * S0.T @ k))
    o, S_T = _fwd(wl, inp.cu_seqlens, a)
    assert _rel(S_T[0, 0], S1) < 1e-14
    assert _rel(o[0], scale * S1.T @ q) < 1e-14
    rng = np.random.default_rng(0)
    dO = rng.standard_normal((1, 3))
    dST = rng.standard_normal((1, 1, 5, 3))
    gr = _bwd(wl, inp.cu_seqlens, a, dO, dST)
    dS1 = scale * np.outer(q, dO[0]) + dST[0, 0]
    kv = S0.T @ k
    dd = dS1.T @ k
    assert _rel(gr["dv"][0], b * dd) < 1e-13
    assert _rel(gr["dS0"][0, 0], g * dS1 - g * b * np.outer(k, dd)) < 1e-13
    db = (v - g * kv) @ dd
    assert abs(gr["dbeta_raw"][0, 0] - db * b * (1 - b)) < 1e-13 * max(1, abs(db))
    dg = (S0 * dS1).sum() - b * kv @ dd
    x = a["alpha"][0, 0] + a["dt_bias"][0]
    dalpha = dg * g * (-np.exp(a["a_log"][0])) / (1 + np.exp(-x))
    assert abs(gr["dalpha"][0, 0] - dalpha) < 1e-13 * max(1, abs(dalpha))
    assert abs(gr["ddt_bias"][0] - dalpha) < 1e-13 * max(1, abs(dalpha))
    # d/d a_log: l = -exp(a_log) softplus(x) so dl/d a_log = l.
    l = np.log(g)
    assert abs(gr["da_log"][0] - dg * g * l) < 1e-13 * max(1, abs(dg * g * l))
    # q/k gradients through the L2 norm (projection onto the normal plane).
    dqh = scale * S1 @ dO[0]
    nq = np.sqrt((a["q"][0] ** 2).sum() + 1e-6)
    assert _rel(gr["dq"][0], (dqh - q * (q @ dqh)) / nq) < 1e-13
    dkh = dS1 @ (b * (v - g * kv)) - g * b * S0 @ dd
    nk = np.sqrt((a["k"][0] ** 2).sum() + 1e-6)
    assert _rel(gr["dk"][0], (dkh - k * (k @ dkh)) / nk) < 1e-13


def test_delta_rule_write_retrieves_value():
    """beta = 1: after one write the state returns, at the written key, rho v + (1 - rho) g S0^T k
    (rho = |k_hat|^2), whatever the decay g -- the error-correcting write of the delta rule."""
    wl, inp, a = _draw(1, 1, 6, 4, (1,), 31)
    a["beta_raw"][:] = np.inf
    o, S_T = _fwd(wl, inp.cu_seqlens, a)
    kraw = a["k"][0]
    khat = kraw / np.sqrt((kraw ** 2).sum() + 1e-6)
    rho = (khat ** 2).sum()
    g = np.exp(-np.exp(a["a_log"][0]) * np.logaddexp(0, a["alpha"][0, 0] + a["dt_bias"][0]))
    want = rho * a["v"][0] + (1 - rho) * g * (a["S0"][0, 0].T @ khat)
    assert _rel(S_T[0, 0].T @ khat, want) < 1e-13
    # With q equal to k the output reads the written value back (o from the updated state).
    a["q"][0] = kraw
    o, _ = _fwd(wl, inp.cu_seqlens, a)
    assert _rel(o[0], want / np.sqrt(6)) < 1e-13


def test_orthogonal_keys_store_and_overwrite():
    """g = 1, beta = 1, S_0 = 0, keys on distinct basis vectors: each key retrieves its value;
    writing a key again replaces (rho-weighted) what it held."""
    wl, inp, a = _draw(1, 1, 8, 3, (6,), 41, S0=False)
    a["beta_raw"][:] = np.inf
    a["a_log"][:] = -np.inf
    keys = [0, 3, 5, 3, 7, 1]
    a["k"][:] = 0.0
    for t, i in enumerate(keys):
        a["k"][t, i] = 1.0
    o, S_T = _fwd(wl, inp.cu_seqlens, a)
    rho = 1.0 / (1.0 + 1e-6)
    S = S_T[0, 0]
    for i in set(keys):
        ts = [t for t, j in enumerate(keys) if j == i]
        want = np.zeros(3)
        for t in ts:
            want = rho * a["v"][t] + (1 - rho) * want
        e = np.zeros(8)
        e[i] = np.sqrt(rho)
        assert _rel(S.T @ e, want) < 1e-12
    for i in set(range(8)) - set(keys):
        assert np.abs(S[i]).max() == 0.0


def test_beta0_gate1_leaves_state_untouched():
    wl, inp, a = _draw(2, 4, 6, 5, (7, 4), 51)
    a["beta_raw"][:] = -np.inf
    a["a_log"][:] = -np.inf
    o, S_T = _fwd(wl, inp.cu_seqlens, a)
    assert np.array_equal(S_T, a["S0"])
    cu = inp.cu_seqlens
    for n in range(2):
        for t in range(cu[n], cu[n + 1]):
            for h in range(4):
                kh = h // 2
                qraw = a["q"][t, kh * 6:(kh + 1) * 6]
                qhat = qraw / np.sqrt((qraw ** 2).sum() + 1e-6)
                assert _rel(o[t, h * 5:(h + 1) * 5], a["S0"][n, h].T @ qhat / np.sqrt(6)) < 1e-14


def test_beta0_decays_state_by_softplus_gate():
    """beta = 0: S_T = S_0 * prod_t g_t with log g = -exp(a_log) * logaddexp(0, alpha + dt_bias)."""
    wl, inp, a = _draw(1, 2, 4, 4, (9,), 61)
    a["beta_raw"][:] = -np.inf
    _, S_T = _fwd(wl, inp.cu_seqlens, a)
    for h in range(2):
        logdecay = (-np.exp(a["a_log"][h]) * np.logaddexp(0, a["alpha"][:, h] + a["dt_bias"][h])).sum()
        assert _rel(S_T[0, h], np.exp(logdecay) * a["S0"][0, h]) < 1e-13


def test_linear_in_values_and_initial_state():
    wl, inp, a = _draw(2, 4, 5, 6, (11, 7), 71)
    rng = np.random.default_rng(3)
    v2 = rng.standard_normal(a["v"].shape)
    S02 = rng.standard_normal(a["S0"].shape)
    o1, s1 = _fwd(wl, inp.cu_seqlens, a)
    b = dict(a, v=v2, S0=S02)
    o2, s2 = _fwd(wl, inp.cu_seqlens, b)
    c = dict(a, v=2.0 * a["v"] - 3.0 * v2, S0=2.0 * a["S0"] - 3.0 * S02)
    o3, s3 = _fwd(wl, inp.cu_seqlens, c)
    assert _rel(o3, 2 * o1 - 3 * o2) < 1e-12
    assert _rel(s3, 2 * s1 - 3 * s2) < 1e-12


def test_query_key_scale_invariance():
    """q_hat and k_hat are normalised: scaling raw q, k by 7 changes o only through the 1e-6 eps."""
    wl, inp, a = _draw(1, 2, 8, 4, (10,), 81)
    o1, _ = _fwd(wl, inp.cu_seqlens, a)
    b = dict(a, q=7.0 * a["q"], k=7.0 * a["k"])
    o2, _ = _fwd(wl, inp.cu_seqlens, b)
    assert _rel(o2, o1) < 1e-6
    c = dict(a, q=2.0 * a["q"])
    # a forgotten normalisation would have doubled o; it must stay put
    o3, _ = _fwd(wl, inp.cu_seqlens, c)
    assert _rel(o3, o1) < 1e-6


def test_shared_key_head_equals_explicit_repeat():
    """v_repeat = 3 with one shared key head == v_repeat = 1 with q/k copied per value head,
    and dq/dk of the shared head == sum of the copies' gradients."""
    wl, inp, a = _draw(2, 6, 4, 5, (8, 5), 91)
    Hk, Hv, Dk = 2, 6, 4
    rep = lambda x: np.concatenate([x[:, (h // 3) * Dk:(h // 3 + 1) * Dk] for h in range(Hv)], 1)
    b = dict(a, q=rep(a["q"]), k=rep(a["k"]))
    wl1 = W.custom(Hk=Hv, Hv=Hv, Dk=Dk, Dv=5, seqlens=(8, 5))
    o, s = _fwd(wl, inp.cu_seqlens, a)
    o1, s1 = _fwd(wl1, inp.cu_seqlens, b)
    assert _rel(o1, o) < 1e-14 and _rel(s1, s) < 1e-14
    rng = np.random.default_rng(5)
    dO = rng.standard_normal(o.shape)
    dS = rng.standard_normal(s.shape)
    g = _bwd(wl, inp.cu_seqlens, a, dO, dS)
    g1 = _bwd(wl1, inp.cu_seqlens, b, dO, dS)
    for key in ("dv", "dalpha", "dbeta_raw", "da_log", "ddt_bias", "dS0"):
        assert _rel(g1[key], g[key]) < 1e-13, key
    for key in ("dq", "dk"):
        summed = np.concatenate([sum(g1[key][:, h * Dk:(h + 1) * Dk] for h in range(kh * 3, kh * 3 + 3))
                                 for kh in range(Hk)], 1)
        assert _rel(summed, g[key]) < 1e-13, key


def test_modulo_head_map_equals_consecutive_map_on_permuted_heads():
    """head_map 1 (value head h reads key head h % Hk) on some inputs == head_map 0 (key
    head h // r) on the same inputs with the value heads renumbered: consecutive head
    j = kh * r + i is modulo head kh + i * Hk.  Every per-head output is the renumbered
    one and dq/dk (each key head's sum over its value heads, in the same order) agree."""
    Hk, Hv, Dk, Dv, r = 2, 6, 4, 5, 3
    wl, inp, a = _draw(Hk, Hv, Dk, Dv, (7, 4), 97)
    perm = np.array([(j % r) * Hk + j // r for j in range(Hv)])   # modulo head of head j
    cols = lambda x, D: np.concatenate([x[:, h * D:(h + 1) * D] for h in perm], 1)
    b = dict(a, v=cols(a["v"], Dv), alpha=a["alpha"][:, perm], beta_raw=a["beta_raw"][:, perm],
             a_log=a["a_log"][perm], dt_bias=a["dt_bias"][perm], S0=a["S0"][:, perm])
    o, s = _fwd(wl, inp.cu_seqlens, a, head_map=1)
    o1, s1 = _fwd(wl, inp.cu_seqlens, b, head_map=0)
    assert np.array_equal(o1, cols(o, Dv)) and np.array_equal(s1, s[:, perm])
    rng = np.random.default_rng(7)
    dO = rng.standard_normal(o.shape)
    dS = rng.standard_normal(s.shape)
    g = _bwd(wl, inp.cu_seqlens, a, dO, dS, head_map=1)
    g1 = _bwd(wl, inp.cu_seqlens, b, cols(dO, Dv), dS[:, perm], head_map=0)
    assert np.array_equal(g1["dv"], cols(g["dv"], Dv))
    for key in ("dalpha", "dbeta_raw"):
        assert np.array_equal(g1[key], g[key][:, perm]), key
    for key in ("da_log", "ddt_bias"):
        assert np.array_equal(g1[key], g[key][perm]), key
    assert np.array_equal(g1["dS0"], g["dS0"][:, perm])
    for key in ("dq", "dk"):
        assert np.array_equal(g1[key], g[key]), key
    # and the two maps do differ on these inputs
    o0, _ = _fwd(wl, inp.cu_seqlens, a, head_map=0)
    assert not np.allclose(o0, o)


def test_heads_and_sequences_are_independent():
    wl, inp, a = _draw(2, 2, 4, 3, (6, 9), 101)
    o, s = _fwd(wl, inp.cu_seqlens, a)
    cu = inp.cu_seqlens
    for n in range(2):
        for h in range(2):
            sl = slice(cu[n], cu[n + 1])
            part = dict(q=a["q"][sl, h * 4:(h + 1) * 4], k=a["k"][sl, h * 4:(h + 1) * 4],
                        v=a["v"][sl, h * 3:(h + 1) * 3], alpha=a["alpha"][sl, h:h + 1],
                        beta_raw=a["beta_raw"][sl, h:h + 1], a_log=a["a_log"][h:h + 1],
                        dt_bias=a["dt_bias"][h:h + 1], S0=a["S0"][n:n + 1, h:h + 1])
            wl1 = W.custom(Hk=1, Hv=1, Dk=4, Dv=3, seqlens=(cu[n + 1] - cu[n],))
            o1, s1 = _fwd(wl1, np.array([0, cu[n + 1] - cu[n]], np.int32), part)
            assert np.array_equal(o1, o[sl, h * 3:(h + 1) * 3])
            assert np.array_equal(s1[0, 0], s[n, h])


def test_zero_upstream_gives_zero_gradients():
    wl, inp, a = _draw(2, 4, 4, 4, (7, 5), 111)
    g = _bwd(wl, inp.cu_seqlens, a, np.zeros((12, 16)), None)
    for key, val in g.items():
        assert np.abs(val).max() == 0.0, key


def test_thread_count_does_not_change_results():
    wl, inp, a = _draw(2, 6, 4, 4, (9, 4, 12), 121)
    rng = np.random.default_rng(1)
    dO = rng.standard_normal((25, 24))
    kw = dict(Hk=2, Hv=6, Dk=4, Dv=4)
    args = (a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"], a["a_log"], a["dt_bias"],
            inp.cu_seqlens)
    g1 = oracle.backward(*args, dO, a["S0"], None, n_threads=1, **kw)
    g8 = oracle.backward(*args, dO, a["S0"], None, n_threads=8, **kw)
    for key in g1:
        assert np.array_equal(g1[key], g8[key]), key


def test_chunk_states_match_forward_prefixes():
    """The state saved at the start of chunk j equals S_T of the sequence cut before it."""
    wl, inp, a = _draw(1, 2, 4, 4, (37, 16), 131)
    o, S_T, states = _fwd(wl, inp.cu_seqlens, a, chunk=16)
    off = oracle.chunk_offsets(inp.cu_seqlens, 16)
    assert list(off) == [0, 3, 4]
    cu = inp.cu_seqlens
    for n in range(2):
        for j in range(off[n + 1] - off[n]):
            cut = cu[n] + 16 * j
            part = {f: (a[f][cu[n]:cut] if f in ("q", "k", "v", "alpha", "beta_raw") else a[f])
                    for f in FIELDS}
            part["S0"] = a["S0"][n:n + 1]
            _, s = _fwd(wl, np.array([0, cut - cu[n]], np.int32), part)
            assert _rel(states[off[n] + j], s[0]) < 1e-14


@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunked_restatement_equals_token_oracle(C):
    wl, inp, a = _draw(2, 6, 8, 12, (37, 0, 100), 141)
    kw = dict(Hk=2, Hv=6, Dk=8, Dv=12)
    rng = np.random.default_rng(7)
    dO = rng.standard_normal((137, 72))
    dS_T = rng.standard_normal((3, 6, 8, 12))
    args = (a["q"], a["k"], a["v"], a["alpha"], a["beta_raw"], a["a_log"], a["dt_bias"],
            inp.cu_seqlens)
    o, s = oracle.forward(*args, a["S0"], **kw)
    oc, sc = chunked.forward(*args, a["S0"], chunk=C, **kw)
    assert _rel(oc, o) < 1e-12 and _rel(sc, s) < 1e-12
    g = oracle.backward(*args, dO, a["S0"], dS_T, **kw)
    gc = chunked.backward(*args, dO, a["S0"], dS_T, chunk=C, **kw)
    for key in g:
        assert _rel(gc[key], g[key]) < 1e-11, key


def test_chunked_restatement_on_tiny_workload_with_chunk16():
    """The tiny fp32 workload (64 tokens) at chunk 16 crosses three chunk boundaries."""
    inp = W.generate(W.get("tiny_f32"))
    f, b = oracle.run_inputs(inp)
    wl = inp.wl
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv)
    args = (inp.q, inp.k, inp.v, inp.alpha, inp.beta_raw, inp.a_log, inp.dt_bias, inp.cu_seqlens)
    oc, sc = chunked.forward(*args, inp.S0, chunk=16, **kw)
    assert _rel(oc, f["o"]) < 1e-12
    gc = chunked.backward(*args, inp.dO, inp.S0, inp.dS_T, chunk=16, **kw)
    for key in b:
        assert _rel(gc[key], b[key]) < 1e-11, key


def test_chunk_maps_scan_to_the_token_oracles_chunk_states():
    """Chunk maps (Phi, R) reproduce a chunk's end state from any start state; their
    log-depth scan gives the token oracle's state at every chunk start; the transposed
    maps carry dS back to the token oracle's dS_0."""
    C = 16
    wl, inp, a = _draw(1, 2, 8, 6, (75,), 101)
    cu = inp.cu_seqlens
    o, S_T, states = _fwd(wl, cu, a, chunk=C)
    rng = np.random.default_rng(8)
    dO = rng.standard_normal(o.shape)
    dS_T = rng.standard_normal(S_T.shape)
    g = _bwd(wl, cu, a, dO, dS_T)
    scale = 1.0 / np.sqrt(8)
    for h in range(2):
        maps, carries = [], []
        for t0 in range(0, 75, C):
            t1 = min(t0 + C, 75)
            Q, _ = chunked._l2(a["q"][t0:t1, :8])
            K, _ = chunked._l2(a["k"][t0:t1, :8])
            V = a["v"][t0:t1, h * 6:(h + 1) * 6]
            b, _, l = chunked._gates(a["alpha"][t0:t1, h], a["beta_raw"][t0:t1, h],
                                     a["a_log"][h], a["dt_bias"][h])
            G = np.cumsum(l)
            maps.append(chunked.chunk_map(Q, K, V, b, G, scale))
            carries.append(chunked.chunk_carry_term(Q, K, V, b, G, scale,
                                                    dO[t0:t1, h * 6:(h + 1) * 6]))
            S = rng.standard_normal((8, 6))
            _, S_next, _ = chunked.chunk_forward(Q, K, V, b, G, S, scale)
            Phi, R = maps[-1]
            assert _rel(Phi @ S + R, S_next) < 1e-13
        starts = chunked.scan_start_states(maps, a["S0"][0, h])
        assert len(starts) == len(maps) == states.shape[0]
        for c, S in enumerate(starts):
            assert _rel(S, states[c, h]) < 1e-12, c
        Phi, R = maps[-1]
        assert _rel(Phi @ starts[-1] + R, S_T[0, h]) < 1e-12
        d = dS_T[0, h]
        for (Phi, _), Gc in zip(reversed(maps), reversed(carries)):
            d = Phi.T @ d + Gc
        assert _rel(d, g["dS0"][0, h]) < 1e-12
