"""Pins of the oracle's neighbour steps (causal depthwise conv1d + SiLU, gated RMSNorm)
to facts other than their own code (no GPU needed):

* central finite differences of each forward pin every gradient of its backward;
* the conv with one tap is an elementwise SiLU(w x); the conv whose only tap is the
  oldest one is a delay line that reads zero before every sequence start (so a
  reversed tap order or a buffer that leaks across sequences fails);
* the norm of a constant row c 1 is c / sqrt(c^2 + eps) times gamma SiLU(z) for any
  row length (so a sum in place of the mean, or eps outside the square root, fails),
  and with eps = 0 the norm does not change when o is scaled.
"""
import numpy as np
import pytest

import oracle


def silu(x):
    return x / (1.0 + np.exp(-x))


def _fd(f, x, h=1e-6):
    """Central differences of the scalar f at x (any shape)."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


def _rel(a, b):
    den = np.abs(b).max()
    return np.abs(a - b).max() / (den if den > 0 else 1.0)


@pytest.mark.parametrize("K,cu", [(4, [0, 5, 9]), (2, [0, 7]), (3, [0, 1, 1, 6])])
def test_conv_gradients_match_central_differences(K, cu):
    rng = np.random.default_rng(K)
    T, C = cu[-1], 3
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, K))
    dy = rng.standard_normal((T, C))
    dx, dw = oracle.conv1d_silu_backward(x, w, cu, dy)
    loss_x = lambda xx: float((oracle.conv1d_silu_forward(xx, w, cu) * dy).sum())
    loss_w = lambda ww: float((oracle.conv1d_silu_forward(x, ww, cu) * dy).sum())
    assert _rel(dx, _fd(loss_x, x)) < 1e-7
    assert _rel(dw, _fd(loss_w, w)) < 1e-7


def test_conv_with_one_tap_is_elementwise_silu():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 5))
    w = rng.standard_normal((5, 1))
    y = oracle.conv1d_silu_forward(x, w, [0, 4, 9])
    assert np.allclose(y, silu(x * w[:, 0]), rtol=0, atol=1e-15)


def test_conv_oldest_tap_is_a_delay_line_reset_at_sequence_starts():
    rng = np.random.default_rng(2)
    K, cu = 3, [0, 5, 6, 10]
    x = rng.standard_normal((10, 2))
    w = np.zeros((2, K))
    w[:, 0] = 1.0                           # only the tap K-1 tokens back
    y = oracle.conv1d_silu_forward(x, w, cu)
    want = np.zeros_like(x)
    for n in range(len(cu) - 1):
        for t in range(cu[n], cu[n + 1]):
            if t - (K - 1) >= cu[n]:
                want[t] = silu(x[t - (K - 1)])
    assert np.array_equal(y, want)


@pytest.mark.parametrize("H,D,eps", [(2, 8, 1e-6), (3, 4, 0.0), (1, 16, 1e-2)])
def test_norm_gradients_match_central_differences(H, D, eps):
    rng = np.random.default_rng(D)
    T = 4
    o = rng.standard_normal((T, H * D))
    z = rng.standard_normal((T, H * D))
    g = rng.standard_normal(D)
    dy = rng.standard_normal((T, H * D))
    d_o, dz, dg = oracle.gated_rmsnorm_backward(o, z, g, dy, H, D, eps)
    f = lambda oo, zz, gg: float((oracle.gated_rmsnorm_forward(oo, zz, gg, H, D, eps) * dy).sum())
    assert _rel(d_o, _fd(lambda oo: f(oo, z, g), o)) < 1e-7
    assert _rel(dz, _fd(lambda zz: f(o, zz, g), z)) < 1e-7
    assert _rel(dg, _fd(lambda gg: f(o, z, gg), g)) < 1e-7


@pytest.mark.parametrize("D", [1, 4, 32])
def test_norm_of_a_constant_row(D):
    rng = np.random.default_rng(3)
    c, eps = -1.7, 0.3
    o = np.full((2, D), c)
    z = rng.standard_normal((2, D))
    g = rng.standard_normal(D)
    y = oracle.gated_rmsnorm_forward(o, z, g, 1, D, eps)
    assert np.allclose(y, c / np.sqrt(c * c + eps) * g * silu(z), rtol=1e-14, atol=0)


def test_norm_is_scale_invariant_without_eps():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((3, 2 * 8))
    z = rng.standard_normal((3, 16))
    g = rng.standard_normal(8)
    y1 = oracle.gated_rmsnorm_forward(o, z, g, 2, 8, 0.0)
    y2 = oracle.gated_rmsnorm_forward(37.5 * o, z, g, 2, 8, 0.0)
    assert _rel(y2, y1) < 1e-14
