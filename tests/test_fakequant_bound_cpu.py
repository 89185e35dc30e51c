"""The fake-quantization tolerances on the CPU: an fp32 emulation of the kernels' arithmetic and order
stays inside them against the fp64 oracle on the GPU tests' cases, and planted mistakes in the
emulation break them (CPU only)."""

import numpy as np
import pytest

from oracle import fakequant_oracle as F
from tests import parity_bound as PB

CASES = [(1, 64, 1.0, False), (37, 320, 0.5, True), (256, 4096, 2.0, False), (3, 128, 0.05, True), (64, 512, 0.2, False)]


def _inputs(n, k, zero_group, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((n, k)) * 0.1).astype(np.float32)
    if zero_group:
        W[0, :64] = 0.0
    alpha = rng.standard_normal((n, k // 64, 4)).astype(np.float32)
    u = rng.uniform(0.01, 0.99, size=(n, k // 64, 4)).astype(np.float32)
    G = rng.standard_normal((n, k)).astype(np.float32)
    return W, alpha, u, G


def _ratios(W, alpha, u, tau, G, **mistake):
    fw, da = PB.emulate_fakequant(W, alpha, u, tau, G, **mistake)
    ref = F.forward(W, alpha.astype(np.float64), u.astype(np.float64), tau)
    _, da_ref = F.backward(W, alpha.astype(np.float64), u.astype(np.float64), tau, G)
    tol, tol_a = PB.fakequant_tolerances(W, tau, G)
    return (np.abs(fw - ref) / tol).max(), (np.abs(da - da_ref) / tol_a).max()


@pytest.mark.parametrize("n,k,tau,zero_group", CASES)
def test_emulated_fakequant_within_tolerance(n, k, tau, zero_group):
    W, alpha, u, G = _inputs(n, k, zero_group, seed=n * 31 + k)
    rf, ra = _ratios(W, alpha, u, tau, G)
    assert rf <= 1.0 and ra <= 1.0, (rf, ra)


@pytest.mark.parametrize("mistake", ["tau_multiplies", "offset_half_range", "D_without_G"])
def test_planted_mistakes_break_the_tolerance(mistake):
    W, alpha, u, G = _inputs(37, 320, True, seed=11)
    rf, ra = _ratios(W, alpha, u, 0.5, G, **{mistake: True})
    assert max(rf, ra) > 1.0, (rf, ra)
