"""Pins of the fake-quantization oracle (CPU)."""

import numpy as np

from oracle import fakequant_oracle as F
from oracle import quant_oracle as Q


def _case(seed, n=6, k=256):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((n, k)) * 0.1).astype(np.float32)
    alpha = rng.standard_normal((n, k // 64, 4))
    u = rng.uniform(0.05, 0.95, size=(n, k // 64, 4))
    return rng, W, alpha, u


def test_one_hot_mixture_is_that_level():
    """A logit far above the others (tau 1) makes the mixture that bit-width's levels."""
    _, W, alpha, u = _case(1)
    for i, b in enumerate(F.BITS):
        a = np.zeros_like(alpha)
        a[..., i] = 1000.0
        got = F.forward(W, a, u, 1.0)
        assert np.array_equal(got, F.levels(W)[i].astype(np.float64))


def test_levels_are_the_round_to_nearest_grid():
    """Each level is s (q - c) with q the nearest code: within half a step of w, on the grid, and equal
    to w where w already is a grid point whose group reaches both ends."""
    rng, W, _, _ = _case(2)
    L = F.levels(W)
    for i, b in enumerate(F.BITS):
        c = ((1 << b) - 1) / 2.0
        mx = np.abs(W.astype(np.float64)).reshape(W.shape[0], -1, 64).max(axis=2)
        s = np.repeat(mx / c, 64, axis=1)
        assert np.all(np.abs(L[i] - W) <= s / 2 * (1 + 1e-5) + 1e-12)
        q = L[i] / s + c
        assert np.allclose(q, np.rint(q), atol=1e-4)
    g = np.zeros((1, 64), np.float32)   # 2-bit grid points with max 1.5 s at s = 0.5: -0.75, -0.25, 0.25, 0.75
    g[0, :4] = [-0.75, -0.25, 0.25, 0.75]
    assert np.array_equal(F.levels(g)[1][0, :4], g[0, :4])
    assert not F.levels(np.zeros((1, 64), np.float32)).any()


def test_levels_match_the_round_to_nearest_encoder_values():
    """The 8-bit level is the dequantized round-to-nearest encoding up to one step: the encoder rounds
    its scale to fp16, which can move a code by one where w sits near a rounding boundary."""
    _, W, _, _ = _case(3)
    bits = np.full((W.shape[0], W.shape[1] // 64), 8, np.uint8)
    codes, scales = Q.quantize_rtn(W, bits)
    from oracle import vbq_oracle as O
    enc = O.dequant(codes, bits, scales)
    step = np.repeat(np.abs(W).reshape(W.shape[0], -1, 64).max(axis=2) / 127.5, 64, axis=1)
    d = np.abs(F.levels(W)[3] - enc)
    assert np.all(d <= step * 1.01)


def test_gradient_matches_finite_differences():
    """dalpha against central differences of L = sum G * forward (a smooth function of alpha)."""
    rng, W, alpha, u = _case(4, n=2, k=128)
    G = rng.standard_normal(W.shape)
    tau = 0.7
    dW, da = F.backward(W, alpha, u, tau, G)
    assert np.array_equal(dW, G)
    h = 1e-6
    num = np.zeros_like(alpha)
    for idx in np.ndindex(alpha.shape):
        ap, am = alpha.copy(), alpha.copy()
        ap[idx] += h
        am[idx] -= h
        num[idx] = ((G * F.forward(W, ap, u, tau)).sum() - (G * F.forward(W, am, u, tau)).sum()) / (2 * h)
    assert np.allclose(da, num, rtol=1e-6, atol=1e-8)


def test_mixture_sums_to_one_and_tau_sharpens():
    _, _, alpha, u = _case(5)
    p1 = F.mixture(alpha, u, 1.0)
    p2 = F.mixture(alpha, u, 0.05)
    assert np.allclose(p1.sum(-1), 1.0) and np.allclose(p2.sum(-1), 1.0)
    assert (p2.max(-1) >= p1.max(-1) - 1e-12).all()
