"""Pin checks for the oracle, written against independent definitions.

Each check takes the functions under test as arguments, so that
test_oracle_mutations.py can run the same checks against deliberately broken
copies and show that every planted mistake is caught.

The independent sides are:
* exact rational arithmetic (fractions.Fraction) from the grid formula;
* closed forms for 1-bit and 8-bit groups;
* a one-hot identity;
* exact power-of-two linearity;
* storage invariants.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

from synth import bf16_bits_to_f32, f32_to_bf16_bits

GROUP = 64


def exact_weight(q: int, b: int, s_bits: int) -> Fraction:
    """The grid value s * (q - (2^b - 1)/2) as an exact rational."""
    s = Fraction(float(np.uint16(s_bits).view(np.float16)))
    return s * (Fraction(q) - Fraction((1 << b) - 1, 2))


def exact_x(x_bits: int) -> Fraction:
    return Fraction(float(bf16_bits_to_f32(np.array([x_bits], np.uint16))[0]))


def tiny_case(seed: int = 0):
    """4 x 128 matrix that visits every 1- and 2-bit code and all four widths."""
    rng = np.random.default_rng(seed)
    widths = np.array([[1, 2], [2, 1], [4, 8], [8, 4]], dtype=np.uint8)
    n, g = widths.shape
    codes = np.zeros((n, g * GROUP), dtype=np.uint8)
    for r in range(n):
        for j in range(g):
            b = int(widths[r, j])
            if b <= 4:
                vals = (np.arange(GROUP) * (r + 1) + j) % (1 << b)
            else:
                vals = rng.integers(0, 256, GROUP)
            codes[r, j * GROUP:(j + 1) * GROUP] = vals
    scales = rng.uniform(0.01, 0.05, size=(n, g)).astype(np.float16).view(np.uint16)
    x = f32_to_bf16_bits(rng.standard_normal(g * GROUP).astype(np.float32))
    return codes, widths, scales, x


def check_dequant_bruteforce(dequant, seed: int = 0) -> None:
    codes, bits, scales, _ = tiny_case(seed)
    W = dequant(codes, bits, scales)
    assert W.dtype == np.float32
    n, k = codes.shape
    for r in range(n):
        for c in range(k):
            g = c // GROUP
            want = exact_weight(int(codes[r, c]), int(bits[r, g]), int(scales[r, g]))
            assert Fraction(float(W[r, c])) == want, (r, c)


def check_gemv_bruteforce(gemv, seed: int = 0) -> None:
    codes, bits, scales, x = tiny_case(seed)
    y = gemv(codes, bits, scales, x)
    n, k = codes.shape
    xs = [exact_x(int(v)) for v in x]
    for r in range(n):
        terms = [exact_weight(int(codes[r, c]), int(bits[r, c // GROUP]), int(scales[r, c // GROUP])) * xs[c]
                 for c in range(k)]
        want = sum(terms, Fraction(0))
        mag = float(sum(abs(t) for t in terms))
        assert abs(float(y[r]) - float(want)) <= 1e-13 * mag + 1e-300, (r, float(y[r]), float(want))


def _rand_matrix(n, g, b, seed):
    rng = np.random.default_rng(seed)
    bits = np.full((n, g), b, np.uint8)
    codes = rng.integers(0, 1 << b, size=(n, g * GROUP)).astype(np.uint8)
    scales = rng.uniform(0.01, 0.05, size=(n, g)).astype(np.float16).view(np.uint16)
    x = f32_to_bf16_bits(rng.standard_normal(g * GROUP).astype(np.float32))
    return codes, bits, scales, x


def check_closed_form_1bit(gemv, seed: int = 1) -> None:
    """All-1-bit rows: y = sum_g (s_g / 2) * sum_k sign(q_k) x_k with sign(1)=+1, sign(0)=-1."""
    n, g = 5, 6
    codes, bits, scales, x = _rand_matrix(n, g, 1, seed)
    xf = bf16_bits_to_f32(x).astype(np.float64).reshape(g, GROUP)
    s = scales.view(np.float16).astype(np.float64)
    sign = np.where(codes.reshape(n, g, GROUP) == 1, 1.0, -1.0)
    want = ((s / 2.0) * (sign * xf[None]).sum(axis=2)).sum(axis=1)
    y = gemv(codes, bits, scales, x)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def check_closed_form_8bit(gemv, seed: int = 2) -> None:
    """All-8-bit rows: y = sum_g s_g (sum_k (q_k - 128) x_k + 0.5 sum_k x_k), int8-grid identity."""
    n, g = 5, 6
    codes, bits, scales, x = _rand_matrix(n, g, 8, seed)
    xf = bf16_bits_to_f32(x).astype(np.float64).reshape(g, GROUP)
    s = scales.view(np.float16).astype(np.float64)
    q8 = codes.reshape(n, g, GROUP).astype(np.int64) - 128   # int8 grid value
    want = (s * ((q8 * xf[None]).sum(axis=2) + 0.5 * xf.sum(axis=1)[None])).sum(axis=1)
    y = gemv(codes, bits, scales, x)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def check_onehot_identity(gemv, seed: int = 3) -> None:
    """s = 1, b = 8, x = e_k: y = q[:, k] - 127.5 exactly (codes round-trip)."""
    n, g = 7, 3
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(n, g * GROUP)).astype(np.uint8)
    bits = np.full((n, g), 8, np.uint8)
    scales = np.full((n, g), 0x3C00, np.uint16)   # fp16 1.0
    for k in (0, 63, 64, 130, g * GROUP - 1):
        x = np.zeros(g * GROUP, np.uint16)
        x[k] = 0x3F80                                  # bf16 1.0
        y = gemv(codes, bits, scales, x)
        assert np.array_equal(y, codes[:, k].astype(np.float64) - 127.5), k


def check_linearity(gemv, seed: int = 4) -> None:
    """y(2^j x) = 2^j y(x) exactly: power-of-two scaling commutes with every rounding."""
    rng = np.random.default_rng(seed)
    n, g = 6, 4
    bits = rng.choice(np.array([1, 2, 4, 8], np.uint8), size=(n, g))
    codes = (rng.integers(0, 256, size=(n, g * GROUP)) &
             ((1 << np.repeat(bits, GROUP, axis=1).astype(np.int64)) - 1)).astype(np.uint8)
    scales = rng.uniform(0.01, 0.05, size=(n, g)).astype(np.float16).view(np.uint16)
    x = f32_to_bf16_bits(rng.standard_normal(g * GROUP).astype(np.float32))
    y = gemv(codes, bits, scales, x)
    for j in (-3, 1, 5):
        xj = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        assert np.array_equal(gemv(codes, bits, scales, xj), y * 2.0 ** j), j


def check_storage(storage_bytes, seed: int = 5) -> None:
    rng = np.random.default_rng(seed)
    bits = rng.choice(np.array([1, 2, 4, 8], np.uint8), size=(33, 17))
    st = storage_bytes(bits)
    counts = {b: int((bits == b).sum()) for b in (1, 2, 4, 8)}
    # a group of 64 codes at b bits fills 8*b bytes
    want = 8 * counts[1] + 16 * counts[2] + 32 * counts[4] + 64 * counts[8]
    assert st["code_bytes"] == want
    assert st["weights"] == bits.size * 64
    assert abs(st["mean_bits"] - want * 8 / (bits.size * 64)) < 1e-15


def check_row_norms_bruteforce(row_norms, seed: int = 0) -> None:
    """||W_r||_2^2 against the exact rational sum of squares of the grid values."""
    codes, bits, scales, _ = tiny_case(seed)
    got = row_norms(codes, bits, scales)
    n, k = codes.shape
    for r in range(n):
        ss = sum((exact_weight(int(codes[r, c]), int(bits[r, c // GROUP]), int(scales[r, c // GROUP])) ** 2
                  for c in range(k)), Fraction(0))
        assert abs(float(got[r]) ** 2 - float(ss)) <= 1e-13 * float(ss) + 1e-300, (r, float(got[r]), float(ss))


def row_norms_hand_case():
    """Three 64-wide rows whose norms are known by hand.

    row 0: b = 2, s = 1, sixteen each of q = 0, 1, 2, 3: w = -1.5, -0.5, 0.5, 1.5,
           sum w^2 = 16 * (2.25 + 0.25 + 0.25 + 2.25) = 80.
    row 1: b = 1, s = 2: every w = +-1, sum w^2 = 64.
    row 2: b = 8, s = 0: every w = 0.
    """
    codes = np.zeros((3, GROUP), np.uint8)
    codes[0] = np.tile(np.arange(4, dtype=np.uint8), 16)
    codes[1] = np.arange(GROUP, dtype=np.uint8) % 2
    codes[2] = np.arange(GROUP, dtype=np.uint8)
    bits = np.array([[2], [1], [8]], np.uint8)
    scales = np.array([[0x3C00], [0x4000], [0x0000]], np.uint16)   # fp16 1.0, 2.0, 0.0
    return codes, bits, scales, np.array([np.sqrt(80.0), 8.0, 0.0])


def check_row_norms_hand(row_norms) -> None:
    codes, bits, scales, want = row_norms_hand_case()
    got = row_norms(codes, bits, scales)
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0.0)
