"""Pins of the oracle's state map (context parallelism) to facts other than its own code:

* the forward's final state is affine in S_0 with that matrix: forward(S_0).S_T =
  Phi S_0 + forward(0).S_T (the forward is pinned on its own);
* the maps of two consecutive pieces of a sequence compose: Phi(a + b) = Phi(b) Phi(a);
* the backward's dS_0 is linear in dS_T with the transposed matrix:
  dS_0(dS_T) = Phi^T dS_T + dS_0(0) (the backward is pinned on its own);
* closed forms: beta = 0 gives exp(sum of log-decays) I; one token with g = 1 and
  beta = 1 gives the projector I - k_hat k_hat^T (idempotent, annihilates k_hat).
A transposed update, a dropped gate or beta, or the wrong token order fails one of them.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def _case(seed, Hk=1, Hv=2, Dk=8, Dv=5, seqlens=(9, 4), head_map=0):
    wl = W.custom(Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=seqlens, S0_std=0.5, dt_bias_std=0.3,
                  packed=False, seed=seed, head_map=head_map)
    return wl, W.generate(wl)


def _phi(wl, i, **kw):
    return oracle.state_map(i.q, i.k, i.alpha, i.beta_raw, i.a_log, i.dt_bias, i.cu_seqlens,
                            Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, head_map=wl.head_map, **kw)


def _fwd(wl, i, S0, cu=None, rows=slice(None)):
    return oracle.forward(i.q[rows], i.k[rows], i.v[rows], i.alpha[rows], i.beta_raw[rows],
                          i.a_log, i.dt_bias, i.cu_seqlens if cu is None else cu, S0, Hk=wl.Hk,
                          Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv, head_map=wl.head_map)


@pytest.mark.parametrize("Hk,Hv,head_map", [(1, 2, 0), (2, 4, 0), (2, 4, 1)])
def test_final_state_is_affine_in_the_start_state(Hk, Hv, head_map):
    wl, i = _case(1, Hk=Hk, Hv=Hv, head_map=head_map)
    Phi = _phi(wl, i)
    _, R = _fwd(wl, i, None)
    _, S_T = _fwd(wl, i, i.S0)
    assert np.allclose(S_T, np.einsum("nhij,nhjv->nhiv", Phi, i.S0) + R, rtol=0, atol=1e-12)


def test_maps_of_consecutive_pieces_compose():
    wl, i = _case(2, seqlens=(13,))
    Phi = _phi(wl, i)[0]
    m = 5
    cu_a, cu_b = np.array([0, m], np.int32), np.array([0, 13 - m], np.int32)
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk)
    Pa = oracle.state_map(i.q[:m], i.k[:m], i.alpha[:m], i.beta_raw[:m], i.a_log, i.dt_bias, cu_a,
                          **kw)[0]
    Pb = oracle.state_map(i.q[m:], i.k[m:], i.alpha[m:], i.beta_raw[m:], i.a_log, i.dt_bias, cu_b,
                          **kw)[0]
    assert np.allclose(Phi, np.einsum("hij,hjk->hik", Pb, Pa), rtol=0, atol=1e-12)
    assert not np.allclose(Phi, np.einsum("hij,hjk->hik", Pa, Pb), rtol=0, atol=1e-6)


def test_backward_start_gradient_is_linear_with_the_transposed_map():
    wl, i = _case(3, seqlens=(11, 6))
    Phi = _phi(wl, i)
    kw = dict(Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv)
    args = (i.q, i.k, i.v, i.alpha, i.beta_raw, i.a_log, i.dt_bias, i.cu_seqlens, i.dO, i.S0)
    g0 = oracle.backward(*args, None, **kw)
    rng = np.random.default_rng(5)
    dS_T = rng.standard_normal(i.S0.shape)
    g1 = oracle.backward(*args, dS_T, **kw)
    want = np.einsum("nhji,nhjv->nhiv", Phi, dS_T) + g0["dS0"]
    assert np.allclose(g1["dS0"], want, rtol=0, atol=1e-11)


def test_no_write_strength_leaves_pure_decay():
    wl, i = _case(4)
    i.beta_raw[:] = -1e3                     # beta = sigmoid(-1000) = 0 in f64
    Phi = _phi(wl, i)
    x = i.alpha.astype(np.float64) + i.dt_bias.astype(np.float64)[None, :]
    ell = -np.exp(i.a_log.astype(np.float64))[None, :] * np.logaddexp(0.0, x)  # log-decays
    for n in range(len(i.cu_seqlens) - 1):
        s = ell[i.cu_seqlens[n]:i.cu_seqlens[n + 1]].sum(0)
        for h in range(wl.Hv):
            assert np.allclose(Phi[n, h], np.exp(s[h]) * np.eye(wl.Dk), rtol=1e-13, atol=0)


def test_one_full_write_without_decay_is_a_projector():
    wl, i = _case(6, seqlens=(1,))
    i.beta_raw[:] = 60.0                     # beta = 1 in f64
    i.alpha[:] = -1e3                        # softplus = 0: g = 1
    Phi = _phi(wl, i)[0]
    k = i.k[0, :wl.Dk].astype(np.float64)
    kh = k / np.sqrt(k @ k + 1e-6)
    for h in range(wl.Hv):
        assert np.allclose(Phi[h], np.eye(wl.Dk) - np.outer(kh, kh), rtol=0, atol=1e-14)
        assert np.allclose(Phi[h] @ Phi[h], Phi[h], atol=1e-6)   # |k_hat| = 1 - O(1e-6)
