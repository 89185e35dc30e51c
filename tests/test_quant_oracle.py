"""Pins of the divergence oracle and the library's round-to-nearest encoder (CPU)."""

import numpy as np
import pytest

from oracle import quant_oracle as Q
from oracle import vbq_oracle as O
from synth import CONFIG0_PROBS, gen_x


@pytest.fixture(scope="module")
def lib():
    from tests.gpu_util import build_lib
    build_lib()
    import mixed_precision_weight_bit_b300 as V
    return V


def _bits(rng, n, g, probs=CONFIG0_PROBS):
    return rng.choice(list(probs.keys()), size=(n, g), p=list(probs.values())).astype(np.uint8)


def test_weights_on_the_grid_come_back_exactly():
    """A group whose codes reach both ends of its range has max|w| = s c_b exactly, so the encoder
    recovers its scale and codes."""
    rng = np.random.default_rng(1)
    n, k = 40, 256
    bits = _bits(rng, n, k // 64)
    qmax = (1 << bits.astype(np.int64)) - 1
    codes = (rng.random((n, k)) * (np.repeat(qmax, 64, axis=1) + 1)).astype(np.uint8)
    codes[:, ::64] = 0
    codes[:, 1::64] = qmax.astype(np.uint8)
    scales = (np.float16(0.25) * rng.integers(1, 9, size=(n, k // 64)).astype(np.float16)).view(np.uint16)
    W = O.dequant(codes, bits, scales)
    q, s = Q.quantize_rtn(W, bits)
    assert np.array_equal(s, scales) and np.array_equal(q, codes)


def test_error_is_half_a_step():
    rng = np.random.default_rng(2)
    n, k = 64, 512
    bits = _bits(rng, n, k // 64)
    W = rng.standard_normal((n, k)).astype(np.float32) * 0.05
    q, s = Q.quantize_rtn(W, bits)
    back = O.dequant(q, bits, s).astype(np.float64)
    sv = O.f16_bits_to_f64(s)
    c = (np.ldexp(1.0, bits.astype(np.int64)) - 1.0) / 2.0
    exact = np.abs(W.astype(np.float64)).reshape(n, -1, 64).max(axis=2) / c
    tol = np.repeat(sv / 2.0 + c * np.abs(sv - exact), 64, axis=1) * (1 + 1e-12)
    assert np.all(np.abs(back - W) <= tol)


def test_zero_and_one_bit_groups():
    W = np.zeros((2, 128), np.float32)
    W[1, 64:] = np.linspace(-1, 1, 64, dtype=np.float32)
    bits = np.array([[1, 4], [2, 1]], np.uint8)
    q, s = Q.quantize_rtn(W, bits)
    assert not q[0].any() and not s[0].any() and not q[1, :64].any() and s[1, 0] == 0
    # 1 bit: s = 2 max|w|, q = 1 exactly where w > 0 (w / s + 1/2 > 1/2)
    assert np.array_equal(q[1, 64:], (W[1, 64:] > 0).astype(np.uint8))


def test_library_encoder_equals_the_oracle(lib):
    rng = np.random.default_rng(3)
    for n, k, scale in [(33, 128, 1.0), (200, 640, 0.02), (7, 64, 3e-6)]:
        bits = _bits(rng, n, k // 64)
        W = (rng.standard_normal((n, k)) * scale).astype(np.float32)
        W[0, :64] = 0.0
        q1, s1 = lib.vbq_quantize_rtn(W, bits)
        q2, s2 = Q.quantize_rtn(W, bits)
        assert np.array_equal(s1, s2) and np.array_equal(q1, q2)


def test_library_encoder_rejects_bad_input(lib):
    with pytest.raises(lib.VbqError) as e:
        lib.vbq_quantize_rtn(np.zeros((2, 100), np.float32), np.ones((2, 1), np.uint8))
    assert e.value.status == 2
    with pytest.raises(lib.VbqError) as e:
        lib.vbq_quantize_rtn(np.zeros((2, 64), np.float32), np.full((2, 1), 3, np.uint8))
    assert e.value.status == 4
    W = np.zeros((1, 64), np.float32)
    W[0, 5] = np.nan
    with pytest.raises(lib.VbqError) as e:
        lib.vbq_quantize_rtn(W, np.ones((1, 1), np.uint8))
    assert e.value.status == 1


def test_kl_and_flips_closed_forms():
    z = np.array([[0.0, 1.0, -2.0], [3.0, 3.5, 0.0]])
    kl, fl = Q.kl_and_flips(z, z)
    assert np.allclose(kl, 0.0, atol=1e-15) and not fl.any()
    # two classes: P = (1/2, 1/2), Q = softmax(0, log 3) = (1/4, 3/4): KL = 1/2 log 2 + 1/2 log(2/3)
    kl, fl = Q.kl_and_flips(np.array([[0.0, 0.0]]), np.array([[0.0, np.log(3.0)]]))
    assert abs(kl[0] - (0.5 * np.log(2.0) + 0.5 * np.log(2.0 / 3.0))) < 1e-15
    kl, fl = Q.kl_and_flips(np.array([[2.0, 0.0]]), np.array([[0.0, 2.0]]))
    assert fl[0] and kl[0] > 0


def test_dense_chain_on_dequantized_weights_is_the_packed_chain():
    """decode_step over dense matrices equal to the dequantized ones gives the packed chain's logits."""
    from synth import gen_model_matrix, model_tiny
    t = model_tiny()
    mats = {}

    def get(layer, proj):
        if (layer, proj) not in mats:
            m = gen_model_matrix(t, layer, proj, seed=4)
            mats[(layer, proj)] = (m.codes, m.bits, m.scales)
        return mats[(layer, proj)]

    x = gen_x(t.d, seed=5)
    a = O.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, x)
    b = O.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, x,
                      dense=lambda layer, proj: O.dequant(*get(layer, proj)))
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
