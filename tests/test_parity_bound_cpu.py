"""The per-element parity bound on the CPU: the emulated kernel arithmetic stays inside it, and an
expected value moved by twice the bound is rejected (CPU only)."""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import CONFIG0_PROBS, f32_to_bf16_bits, gen_matrix, gen_matrix_with_bits, gen_stress, gen_x
from tests import parity_bound as PB


def _edge_x(k, kind, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "zero":
        return np.zeros(k, np.uint16)
    if kind == "subnormal":   # bf16 subnormals only: |x| < 2^-126
        return f32_to_bf16_bits((rng.uniform(-1, 1, k) * 2.0 ** -127).astype(np.float32))
    if kind == "huge":        # +-2^120 with ordinary values beside them
        v = rng.standard_normal(k).astype(np.float32)
        v[::7] = np.float32(2.0 ** 120) * np.sign(v[::7])
        return f32_to_bf16_bits(v)
    if kind == "cancel":      # each group holds pairs x, -x: sums of equal-code pairs cancel exactly
        v = rng.standard_normal(k // 2).astype(np.float32)
        return f32_to_bf16_bits(np.stack([v, -v], axis=1).reshape(-1))
    return gen_x(k, seed=seed)


CASES = {
    "config0_40x256": lambda: gen_matrix(40, 256, CONFIG0_PROBS, seed=3),
    "all1": lambda: gen_matrix_with_bits(np.full((12, 4), 1, np.uint8), 1, (9, 1)),
    "all2": lambda: gen_matrix_with_bits(np.full((12, 4), 2, np.uint8), 2, (9, 2)),
    "all4": lambda: gen_matrix_with_bits(np.full((12, 4), 4, np.uint8), 3, (9, 4)),
    "all8": lambda: gen_matrix_with_bits(np.full((12, 4), 8, np.uint8), 4, (9, 8)),
    "stress_e": lambda: gen_stress("e", 16, 512),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("xkind", ["normal", "zero", "subnormal", "huge", "cancel"])
def test_emulated_arithmetic_within_bound(name, xkind):
    m = CASES[name]()
    x = _edge_x(m.K, xkind, seed=5)
    ref = O.gemv(m.codes, m.bits, m.scales, x)
    y = PB.emulate_gemv(m.codes, m.bits, m.scales, x)
    bound = PB.gemv_bound(m.codes, m.bits, m.scales, x)
    PB.check_within(y, ref, bound)
    if xkind == "zero":
        assert np.array_equal(y, np.zeros_like(y))


def test_bound_is_tight_against_the_normalized_bar():
    m = gen_matrix(64, 1024, CONFIG0_PROBS, seed=6)
    x = gen_x(m.K, seed=6)
    b = PB.gemv_bound(m.codes, m.bits, m.scales, x)
    norms = O.row_norms(m.codes, m.bits, m.scales)
    xn = np.linalg.norm(O.bf16_bits_to_f64(x))
    assert np.max(b / (norms * xn)) < 1e-4   # more than an order of magnitude below the 2e-3 bar


def test_weakened_expected_value_fails_the_bound():
    m = gen_matrix(40, 256, CONFIG0_PROBS, seed=7)
    x = gen_x(m.K, seed=7)
    ref = O.gemv(m.codes, m.bits, m.scales, x)
    y = PB.emulate_gemv(m.codes, m.bits, m.scales, x)
    bound = PB.gemv_bound(m.codes, m.bits, m.scales, x)
    PB.check_within(y, ref, bound)
    bad = ref.copy()
    bad[17] += 2.0 * bound[17]          # an expected value off by twice the bound in one row
    with pytest.raises(AssertionError):
        PB.check_within(y, bad, bound)
    # the normalized 2e-3 bar alone would not notice it
    norms = O.row_norms(m.codes, m.bits, m.scales)
    assert O.normalized_error(y, bad, norms, x) < 2e-3


def test_tc_bound_covers_fp16_rounding_of_weights_and_x():
    # An fp16 model of the tensor-core arithmetic: w and x * 2^p rounded to fp16, products summed in fp64.
    m = gen_matrix(30, 512, CONFIG0_PROBS, seed=8)
    X = gen_x(m.K, seed=8, batch=3)
    W = O.dequant(m.codes, m.bits, m.scales).astype(np.float16).astype(np.float64)
    Xf = O.bf16_bits_to_f64(X)
    p = 14 - PB.exp_above(np.abs(Xf).max(axis=1))
    Xh = (Xf * np.ldexp(1.0, p)[:, None]).astype(np.float16).astype(np.float64) / np.ldexp(1.0, p)[:, None]
    Y = Xh @ W.T
    ref = O.gemm(m.codes, m.bits, m.scales, X)
    PB.check_within(Y, ref, PB.tc_bound(m.codes, m.bits, m.scales, X))
