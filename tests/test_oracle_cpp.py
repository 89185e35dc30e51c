"""The C++ oracle against the pins and against the numpy oracle (CPU only).

oracle/vbq_oracle.cpp restates the same definitions in plain single-threaded
C++. It has to pass every pin the numpy oracle passes; on the same inputs its
dequantized weights equal the numpy oracle's bit for bit, and its fp64 sums
agree up to the order of summation (the numpy oracle uses a BLAS product).
"""

import shutil

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import (CONFIG0_PROBS, gen_matrix, gen_matrix_with_bits, gen_model_matrix, gen_stress, gen_x,
                   model_tiny)
from tests import oracle_pins as P

pytestmark = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")


@pytest.fixture(scope="module")
def C():
    from oracle import vbq_oracle_cpp
    vbq_oracle_cpp.build()
    return vbq_oracle_cpp


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cpp_dequant_bruteforce_exact(C, seed):
    P.check_dequant_bruteforce(C.dequant, seed)


@pytest.mark.parametrize("seed", [0, 1])
def test_cpp_gemv_bruteforce_exact(C, seed):
    P.check_gemv_bruteforce(C.gemv, seed)


def test_cpp_closed_forms_onehot_linearity(C):
    P.check_closed_form_1bit(C.gemv)
    P.check_closed_form_8bit(C.gemv)
    P.check_onehot_identity(C.gemv)
    P.check_linearity(C.gemv)


@pytest.mark.parametrize("seed", [0, 1])
def test_cpp_row_norms_pins(C, seed):
    P.check_row_norms_bruteforce(C.row_norms, seed)
    P.check_row_norms_hand(C.row_norms)


def _cases():
    yield "config0_300x1024", gen_matrix(300, 1024, CONFIG0_PROBS, seed=3)
    yield "stress_e_256", gen_stress("e", 256, 1024)
    for b in (1, 2, 4, 8):
        yield f"all{b}", gen_matrix_with_bits(np.full((40, 8), b, np.uint8), 5, (9, b))


@pytest.mark.parametrize("name", [n for n, _ in _cases()])
def test_cpp_matches_numpy_oracle(C, name):
    m = dict(_cases())[name]
    Wc, Wn = C.dequant(m.codes, m.bits, m.scales), O.dequant(m.codes, m.bits, m.scales)
    assert np.array_equal(Wc.view(np.uint32), Wn.view(np.uint32))
    x = gen_x(m.K, seed=12)
    yc, yn = C.gemv(m.codes, m.bits, m.scales, x), O.gemv(m.codes, m.bits, m.scales, x)
    # Both sum the same exact fp64 products; only the order differs: K ulps of sum |w x|.
    mag = np.abs(Wn.astype(np.float64)) @ np.abs(O.bf16_bits_to_f64(x))
    assert np.all(np.abs(yc - yn) <= m.K * 2.0 ** -52 * mag)
    nc, nn = C.row_norms(m.codes, m.bits, m.scales), O.row_norms(m.codes, m.bits, m.scales)
    np.testing.assert_allclose(nc, nn, rtol=m.K * 2.0 ** -52, atol=0.0)


def test_cpp_bf16_rounding_matches_numpy(C):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        np.ldexp(1.0 + np.arange(0, 256) / 256.0 + 1.0 / 512.0, -3),   # exact ties
                        np.ldexp(rng.uniform(-1, 1, 100), -130),                        # bf16 subnormals
                        np.array([0.0, -0.0, 1.0, -1.0])])
    assert np.array_equal(C.to_bf16_bits(v), O.f64_to_bf16_bits(v))


def test_cpp_rejects_bad_inputs(C):
    m = gen_matrix(4, 128, CONFIG0_PROBS, seed=1)
    bad_bits = m.bits.copy()
    bad_bits[0, 0] = 3
    with pytest.raises(ValueError):
        C.gemv(m.codes, bad_bits, m.scales, gen_x(128, seed=1))
    bad_codes = m.codes.copy()
    one = np.argwhere(m.bits == 1)[0]
    bad_codes[one[0], one[1] * 64] = 2
    with pytest.raises(ValueError):
        C.dequant(bad_codes, m.bits, m.scales)
    with pytest.raises(ValueError):
        C.row_norms(m.codes[:, :100], m.bits, m.scales)


def test_cpp_decode_step_matches_numpy_chain(C):
    t = model_tiny()
    get = lambda layer, proj: (lambda m: (m.codes, m.bits, m.scales))(gen_model_matrix(t, layer, proj, seed=4))
    x = gen_x(t.d, seed=5)
    ref = O.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, x)
    got = C.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, t.d, t.d_ff, t.vocab, x)
    # The chains differ only in the order of the RMSNorm and dot-product sums (numpy's pairwise and
    # BLAS orders); that can move a bf16 input by one ulp where it sits on a rounding tie.
    head = get(t.n_layers, "head")
    scale = np.max(O.row_norms(*head)) * np.sqrt(t.d)
    assert np.max(np.abs(got - ref)) / scale < 1e-6
