"""Pins of the fake-quantization oracle (CPU).

Each check takes the oracle as M (levels, mixture, forward, backward), so that
test_planted_mistakes_fail_a_pin can run the same checks on copies of the
oracle with one step done the wrong way."""

import types

import numpy as np
import pytest

from oracle import fakequant_oracle as F
from oracle import quant_oracle as Q
from oracle import vbq_oracle as O


def _case(seed, n=6, k=256):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((n, k)) * 0.1).astype(np.float32)
    alpha = rng.standard_normal((n, k // 64, 4))
    u = rng.uniform(0.05, 0.95, size=(n, k // 64, 4))
    return rng, W, alpha, u


def check_one_hot_mixture_is_that_level(M=F):
    """A logit far above the others (tau 1) makes the mixture that bit-width's levels."""
    _, W, alpha, u = _case(1)
    for i, b in enumerate(F.BITS):
        a = np.zeros_like(alpha)
        a[..., i] = 1000.0
        got = M.forward(W, a, u, 1.0)
        assert np.array_equal(got, M.levels(W)[i].astype(np.float64))


def check_levels_are_the_round_to_nearest_grid(M=F):
    """Each level is s (q - c) with q the nearest code: within half a step of w, on the grid, and equal
    to w where w already is a grid point whose group reaches both ends."""
    _, W, _, _ = _case(2)
    L = M.levels(W)
    for i, b in enumerate(F.BITS):
        c = ((1 << b) - 1) / 2.0
        mx = np.abs(W.astype(np.float64)).reshape(W.shape[0], -1, 64).max(axis=2)
        s = np.repeat(mx / c, 64, axis=1)
        assert np.all(np.abs(L[i] - W) <= s / 2 * (1 + 1e-5) + 1e-12)
        q = L[i] / s + c
        assert np.allclose(q, np.rint(q), atol=1e-4)
    g = np.zeros((1, 64), np.float32)   # 2-bit grid points with max 1.5 s at s = 0.5: -0.75, -0.25, 0.25, 0.75
    g[0, :4] = [-0.75, -0.25, 0.25, 0.75]
    assert np.array_equal(M.levels(g)[1][0, :4], g[0, :4])
    assert not M.levels(np.zeros((1, 64), np.float32)).any()


def check_levels_match_the_round_to_nearest_encoder_values(M=F):
    """The 8-bit level is the dequantized round-to-nearest encoding up to one step: the encoder rounds
    its scale to fp16, which can move a code by one where w sits near a rounding boundary."""
    _, W, _, _ = _case(3)
    bits = np.full((W.shape[0], W.shape[1] // 64), 8, np.uint8)
    codes, scales = Q.quantize_rtn(W, bits)
    enc = O.dequant(codes, bits, scales)
    step = np.repeat(np.abs(W).reshape(W.shape[0], -1, 64).max(axis=2) / 127.5, 64, axis=1)
    d = np.abs(M.levels(W)[3] - enc)
    assert np.all(d <= step * 1.01)


def check_gradient_matches_finite_differences(M=F):
    """dalpha against central differences of L = sum G * forward (a smooth function of alpha); dW = G."""
    rng, W, alpha, u = _case(4, n=2, k=128)
    G = rng.standard_normal(W.shape)
    tau = 0.7
    dW, da = M.backward(W, alpha, u, tau, G)
    assert np.array_equal(dW, G)
    h = 1e-6
    num = np.zeros_like(alpha)
    for idx in np.ndindex(alpha.shape):
        ap, am = alpha.copy(), alpha.copy()
        ap[idx] += h
        am[idx] -= h
        num[idx] = ((G * M.forward(W, ap, u, tau)).sum() - (G * M.forward(W, am, u, tau)).sum()) / (2 * h)
    assert np.allclose(da, num, rtol=1e-6, atol=1e-8)


def check_mixture_sums_to_one_and_tau_sharpens(M=F):
    _, _, alpha, u = _case(5)
    p1 = M.mixture(alpha, u, 1.0)
    p2 = M.mixture(alpha, u, 0.05)
    assert np.allclose(p1.sum(-1), 1.0) and np.allclose(p2.sum(-1), 1.0)
    assert (p2.max(-1) >= p1.max(-1) - 1e-12).all()


def check_gumbel_noise_closed_form(M=F):
    """Equal logits at tau 1: exp(-log(-log u)) = 1 / (-log u), so pi_b is proportional to 1 / (-log u_b)."""
    _, _, alpha, u = _case(6)
    p = M.mixture(np.zeros_like(alpha), u, 1.0)
    w = 1.0 / -np.log(u)
    assert np.allclose(p, w / w.sum(-1, keepdims=True), rtol=1e-13, atol=0)


def check_equal_noise_is_softmax_of_logits_over_tau(M=F):
    """The same u for all four widths cancels: pi = softmax(alpha / tau); at alpha = (0, log 2, log 3,
    log 4) and tau 1 that is (1, 2, 3, 4) / 10, and at tau 1/2 (1, 4, 9, 16) / 30."""
    a = np.log(np.array([1.0, 2.0, 3.0, 4.0]))[None, None, :]
    u = np.full((1, 1, 4), 0.3)
    assert np.allclose(M.mixture(a, u, 1.0)[0, 0], [0.1, 0.2, 0.3, 0.4], rtol=1e-14, atol=0)
    assert np.allclose(M.mixture(a, u, 0.5)[0, 0], np.array([1.0, 4.0, 9.0, 16.0]) / 30.0, rtol=1e-14, atol=0)


def check_mixture_of_two_widths_is_their_weighted_levels(M=F):
    """Logits (0, 0, -inf-like, -inf-like) with equal noise split the weight evenly between 1 and 2 bits,
    group by group, whatever the other groups' logits."""
    _, W, alpha, u = _case(7)
    a = alpha.copy()
    a[0, 1] = [0.0, 0.0, -1000.0, -1000.0]
    u2 = u.copy()
    u2[0, 1] = 0.5
    got = M.forward(W, a, u2, 1.0)
    L = M.levels(W).astype(np.float64)
    assert np.allclose(got[0, 64:128], 0.5 * (L[0, 0, 64:128] + L[1, 0, 64:128]), rtol=1e-15, atol=1e-300)


CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__[6:])
def test_pin(check):
    check(F)


# ---- planted mistakes ----

def _levels_variant(kind):
    def levels(W):
        W = np.asarray(W, dtype=np.float32)
        n, k = W.shape
        Wg = W.reshape(n, k // 64, 64)
        if kind == "scale_from_row_max":
            mx = np.repeat(np.abs(W).max(axis=1, keepdims=True)[:, :, None], k // 64, axis=1)
        else:
            mx = np.abs(Wg).max(axis=2, keepdims=True)
        out = np.zeros((4, n, k // 64, 64), np.float32)
        for i, b in enumerate(F.BITS):
            qmax = np.float32((1 << b) - 1)
            c = np.float32(1 << (b - 1)) if kind == "offset_2^b/2" else np.float32(0.5) * qmax
            with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
                s, r = mx / c, c / mx
                x = Wg * r + c
                q = np.clip(np.floor(x) if kind == "codes_floor" else np.rint(x), np.float32(0), qmax)
                v = s * (q - c)
            out[i] = np.where(mx > 0, v, np.float32(0))
        return out.reshape(4, n, k)
    return levels


def _mixture_variant(kind):
    def mixture(alpha, u, tau):
        a, uu = np.asarray(alpha, np.float64), np.asarray(u, np.float64)
        g = -np.log(-np.log(uu))
        if kind == "gumbel_sign":
            g = -g
        if kind == "gumbel_single_log":
            g = -np.log(uu)
        if kind == "tau_on_noise_only":
            z = a + g / tau
        elif kind == "tau_multiplies":
            z = (a + g) * tau
        else:
            z = (a + g) / tau
        axis = -2 if kind == "softmax_over_groups" else -1
        e = np.exp(z - z.max(axis=axis, keepdims=True))
        return e / e.sum(axis=axis, keepdims=True)
    return mixture


def _oracle_with(levels=None, mixture=None, forward_kind=None, backward_kind=None):
    lv = levels or F.levels
    mix = mixture or F.mixture

    def forward(W, alpha, u, tau):
        Qv = lv(W).astype(np.float64)
        pi = mix(alpha, u, tau)
        if forward_kind == "group_index_modulo":
            piw = np.tile(np.moveaxis(pi, -1, 0), (1, 1, 64))   # column j takes group j % G
        else:
            piw = np.repeat(np.moveaxis(pi, -1, 0), 64, axis=2)
        return (piw * Qv).sum(axis=0)

    def backward(W, alpha, u, tau, G):
        Qv = lv(W).astype(np.float64)
        pi = mix(alpha, u, tau)
        n, k = np.asarray(W).shape
        Gd = np.asarray(G, np.float64)
        prod = Qv if backward_kind == "D_without_G" else Gd[None] * Qv
        D = np.moveaxis(prod.reshape(4, n, k // 64, 64).sum(axis=3), 0, -1)
        mean = (pi * D).sum(axis=-1, keepdims=True)
        dW = np.zeros_like(Gd) if backward_kind == "no_straight_through" else Gd.copy()
        if backward_kind == "no_tau":
            return dW, pi * (D - mean)
        if backward_kind == "no_centering":
            return dW, pi / tau * D
        return dW, pi / tau * (D - mean)

    return types.SimpleNamespace(levels=lv, mixture=mix, forward=forward, backward=backward)


MUTANTS = {
    "levels_offset_2^b/2": lambda: _oracle_with(levels=_levels_variant("offset_2^b/2")),
    "levels_scale_from_row_max": lambda: _oracle_with(levels=_levels_variant("scale_from_row_max")),
    "levels_codes_floor": lambda: _oracle_with(levels=_levels_variant("codes_floor")),
    "mixture_gumbel_sign": lambda: _oracle_with(mixture=_mixture_variant("gumbel_sign")),
    "mixture_gumbel_single_log": lambda: _oracle_with(mixture=_mixture_variant("gumbel_single_log")),
    "mixture_tau_on_noise_only": lambda: _oracle_with(mixture=_mixture_variant("tau_on_noise_only")),
    "mixture_tau_multiplies": lambda: _oracle_with(mixture=_mixture_variant("tau_multiplies")),
    "mixture_softmax_over_groups": lambda: _oracle_with(mixture=_mixture_variant("softmax_over_groups")),
    "forward_group_index_modulo": lambda: _oracle_with(forward_kind="group_index_modulo"),
    "backward_no_tau": lambda: _oracle_with(backward_kind="no_tau"),
    "backward_no_centering": lambda: _oracle_with(backward_kind="no_centering"),
    "backward_D_without_G": lambda: _oracle_with(backward_kind="D_without_G"),
    "backward_no_straight_through": lambda: _oracle_with(backward_kind="no_straight_through"),
}


def test_unmutated_copy_passes_every_pin():
    M = _oracle_with(levels=_levels_variant(None), mixture=_mixture_variant(None))
    for check in CHECKS:
        check(M)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    M = MUTANTS[name]()
    failed = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(M)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the mutant {name}"
