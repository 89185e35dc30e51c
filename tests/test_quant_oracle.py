"""Pins of the divergence oracle and the library's round-to-nearest encoder (CPU).

The oracle's pins are checks that take the oracle as M (quantize_rtn,
log_softmax, kl_and_flips), so that test_planted_mistakes_fail_a_pin can run
them on copies of the oracle with one step done the wrong way."""

import types

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


def check_weights_on_the_grid_come_back_exactly(M=Q):
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
    q, s = M.quantize_rtn(W, bits)
    assert np.array_equal(s, scales) and np.array_equal(q, codes)


def check_error_is_half_a_step(M=Q):
    rng = np.random.default_rng(2)
    n, k = 64, 512
    bits = _bits(rng, n, k // 64)
    W = rng.standard_normal((n, k)).astype(np.float32) * 0.05
    q, s = M.quantize_rtn(W, bits)
    back = O.dequant(q, bits, s).astype(np.float64)
    sv = O.f16_bits_to_f64(s)
    c = (np.ldexp(1.0, bits.astype(np.int64)) - 1.0) / 2.0
    exact = np.abs(W.astype(np.float64)).reshape(n, -1, 64).max(axis=2) / c
    tol = np.repeat(sv / 2.0 + c * np.abs(sv - exact), 64, axis=1) * (1 + 1e-12)
    assert np.all(np.abs(back - W) <= tol)


def check_zero_and_one_bit_groups(M=Q):
    W = np.zeros((2, 128), np.float32)
    W[1, 64:] = np.linspace(-1, 1, 64, dtype=np.float32)
    bits = np.array([[1, 4], [2, 1]], np.uint8)
    q, s = M.quantize_rtn(W, bits)
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


def check_kl_and_flips_closed_forms(M=Q):
    z = np.array([[0.0, 1.0, -2.0], [3.0, 3.5, 0.0]])
    kl, fl = M.kl_and_flips(z, z)
    assert np.allclose(kl, 0.0, atol=1e-15) and not fl.any()
    # two classes: P = (1/2, 1/2), Q = softmax(0, log 3) = (1/4, 3/4): KL = 1/2 log 2 + 1/2 log(2/3)
    kl, fl = M.kl_and_flips(np.array([[0.0, 0.0]]), np.array([[0.0, np.log(3.0)]]))
    assert abs(kl[0] - (0.5 * np.log(2.0) + 0.5 * np.log(2.0 / 3.0))) < 1e-15
    kl, fl = M.kl_and_flips(np.array([[2.0, 0.0]]), np.array([[0.0, 2.0]]))
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


def check_codes_are_the_nearest_points_of_the_stored_grid(M=Q):
    """Brute force over every code: the chosen code's value s16 (q - c) is no farther from w than any
    other code's, with s16 the stored fp16 scale (the decoder's grid). The distances are exact in fp64
    (an fp16 scale times a half-integer, minus an fp32 weight)."""
    rng = np.random.default_rng(10)
    n, k = 24, 256
    for bits in (_bits(rng, n, k // 64), np.full((n, k // 64), 8, np.uint8)):
        W = (rng.standard_normal((n, k)) * 0.3).astype(np.float32)
        q, s = M.quantize_rtn(W, bits)
        sv = np.repeat(O.f16_bits_to_f64(s), 64, axis=1)
        b = np.repeat(bits.astype(np.int64), 64, axis=1)
        c = (np.ldexp(1.0, b) - 1.0) / 2.0
        w = W.astype(np.float64)
        best = np.full(w.shape, np.inf)
        for code in range(256):
            ok = code < np.ldexp(1.0, b)
            best = np.where(ok, np.minimum(best, np.abs(sv * (code - c) - w)), best)
        assert np.all(np.abs(sv * (q.astype(np.float64) - c) - w) <= best)


def check_scale_is_the_nearest_fp16_of_the_exact_one(M=Q):
    """The stored scale is no farther from max|w| / c than either fp16 neighbour."""
    rng = np.random.default_rng(11)
    n, k = 40, 512
    bits = _bits(rng, n, k // 64)
    W = (rng.standard_normal((n, k)) * np.exp(rng.uniform(-8, 2, size=(n, 1)))).astype(np.float32)
    _, s = M.quantize_rtn(W, bits)
    c = (np.ldexp(1.0, bits.astype(np.int64)) - 1.0) / 2.0
    exact = np.abs(W.astype(np.float64)).reshape(n, -1, 64).max(axis=2) / c
    sv = O.f16_bits_to_f64(s)
    lo = O.f16_bits_to_f64(np.maximum(s.astype(np.int64) - 1, 0).astype(np.uint16))
    hi = O.f16_bits_to_f64((s.astype(np.int64) + 1).astype(np.uint16))
    assert np.all(np.abs(sv - exact) <= np.abs(lo - exact)) and np.all(np.abs(sv - exact) <= np.abs(hi - exact))


def check_kl_three_classes_and_flip_rule(M=Q):
    """P = (1, 2, 1) / 4 against uniform Q: KL = sum P log(3 P) = log 3 - (3/2) log 2. A flip compares
    only the argmax: (3, 1, 0) against (3, 0, 1) keeps it, (0, 1, 3) against (0, 3, 1) does not."""
    z = np.log(np.array([[1.0, 2.0, 1.0]]))
    kl, fl = M.kl_and_flips(z, np.zeros((1, 3)))
    assert abs(kl[0] - (np.log(3.0) - 1.5 * np.log(2.0))) < 1e-15
    _, fl = M.kl_and_flips(np.array([[3.0, 1.0, 0.0], [0.0, 1.0, 3.0]]), np.array([[3.0, 0.0, 1.0], [0.0, 3.0, 1.0]]))
    assert not fl[0] and fl[1]
    assert np.allclose(M.log_softmax(np.array([0.0, np.log(3.0)])), np.log([0.25, 0.75]), rtol=0, atol=1e-15)


CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__[6:])
def test_pin(check):
    check(Q)


# ---- planted mistakes ----

def _rtn_variant(kind):
    def quantize_rtn(W, bits):
        W = np.asarray(W, dtype=np.float32).astype(np.float64)
        n, k = W.shape
        g = k // 64
        Wg = W.reshape(n, g, 64)
        b = np.asarray(bits, dtype=np.int64)
        c = np.ldexp(1.0, b - 1) if kind == "offset_2^b/2" else (np.ldexp(1.0, b) - 1.0) / 2.0
        qmax = np.ldexp(1.0, b) - 1.0
        mx = np.repeat(np.abs(W).max(axis=1, keepdims=True), g, axis=1) if kind == "scale_over_row" \
            else np.abs(Wg).max(axis=2)
        if kind == "scale_truncated":
            s16 = (mx / c).astype(np.float32).astype(np.float16)
            s16 = np.where(s16.astype(np.float64) > mx / c, np.nextafter(s16, np.float16(0)), s16).astype(np.float16)
        else:
            s16 = (mx / c).astype(np.float16)
        s = mx / c if kind == "codes_from_unrounded_scale" else s16.astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            x = Wg / s[:, :, None] + c[:, :, None]
            q = np.where(s[:, :, None] > 0, np.floor(x) if kind == "codes_floor" else np.rint(x), 0.0)
        q = np.clip(q, 0.0, qmax[:, :, None])
        return q.reshape(n, k).astype(np.uint8), s16.view(np.uint16)
    return quantize_rtn


def _kl_variant(kind):
    def kl_and_flips(dense_logits, test_logits):
        lp, lq = Q.log_softmax(dense_logits), Q.log_softmax(test_logits)
        if kind == "reversed":
            kl = (np.exp(lq) * (lq - lp)).sum(axis=-1)
        elif kind == "unweighted":
            kl = (lp - lq).sum(axis=-1)
        else:
            kl = (np.exp(lp) * (lp - lq)).sum(axis=-1)
        pick = np.argmin if kind == "flips_on_argmin" else np.argmax
        return kl, pick(dense_logits, axis=-1) != pick(test_logits, axis=-1)
    return kl_and_flips


def _log_softmax_no_norm(z):
    z = np.asarray(z, dtype=np.float64)
    return z - z.max(axis=-1, keepdims=True)


def _oracle_with(rtn=None, kl=None, log_softmax=None):
    return types.SimpleNamespace(quantize_rtn=rtn or Q.quantize_rtn, kl_and_flips=kl or Q.kl_and_flips,
                                 log_softmax=log_softmax or Q.log_softmax)


MUTANTS = {
    "rtn_offset_2^b/2": lambda: _oracle_with(rtn=_rtn_variant("offset_2^b/2")),
    "rtn_scale_over_row": lambda: _oracle_with(rtn=_rtn_variant("scale_over_row")),
    "rtn_scale_truncated": lambda: _oracle_with(rtn=_rtn_variant("scale_truncated")),
    "rtn_codes_from_unrounded_scale": lambda: _oracle_with(rtn=_rtn_variant("codes_from_unrounded_scale")),
    "rtn_codes_floor": lambda: _oracle_with(rtn=_rtn_variant("codes_floor")),
    "kl_reversed": lambda: _oracle_with(kl=_kl_variant("reversed")),
    "kl_unweighted": lambda: _oracle_with(kl=_kl_variant("unweighted")),
    "flips_on_argmin": lambda: _oracle_with(kl=_kl_variant("flips_on_argmin")),
    "log_softmax_unnormalised": lambda: _oracle_with(log_softmax=_log_softmax_no_norm),
}


def test_unmutated_copy_passes_every_pin():
    M = _oracle_with(rtn=_rtn_variant(None), kl=_kl_variant(None))
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
