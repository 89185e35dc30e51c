"""Full-size parity on every output element (GPU): the per-element bound of the kernels' arithmetic
(tests/parity_bound.py) and the normalized 2e-3 bar, on the shapes the bench times."""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import CONFIG0_PROBS, f32_to_bf16_bits, gen_matrix, gen_stress, gen_x
from tests import parity_bound as PB
from tests.gpu_util import TOL, dev_u16, gemv_err, gpu_gemm, gpu_gemv, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _check_gemv(V, m, x):
    mat = V.Matrix(m.codes, m.bits, m.scales)
    y = gpu_gemv(V, mat, x)
    mat.close()
    assert np.isfinite(y).all()
    ref = O.gemv(m.codes, m.bits, m.scales, x)
    PB.check_within(y, ref, PB.gemv_bound(m.codes, m.bits, m.scales, x))
    assert gemv_err(m, x, y) <= TOL
    return y


def test_gemv_all_rows_14336x4096(V):
    m = gen_matrix(14336, 4096, CONFIG0_PROBS, seed=0)
    _check_gemv(V, m, gen_x(m.K, seed=3))


@pytest.mark.parametrize("case", ["a", "b", "c", "d", "e"])
def test_gemv_all_rows_stress_8192(V, case):
    m = gen_stress(case, 8192, 8192)
    _check_gemv(V, m, gen_x(m.K, seed=21))


def _edge_x(k, kind, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "zero":
        return np.zeros(k, np.uint16)
    if kind == "subnormal":
        return f32_to_bf16_bits((rng.uniform(-1, 1, k) * 2.0 ** -127).astype(np.float32))
    if kind == "huge":
        v = rng.standard_normal(k).astype(np.float32)
        v[::7] = np.float32(2.0 ** 120) * np.sign(v[::7])
        return f32_to_bf16_bits(v)
    v = rng.standard_normal(k // 2).astype(np.float32)   # "cancel": x, -x pairs
    return f32_to_bf16_bits(np.stack([v, -v], axis=1).reshape(-1))


@pytest.mark.parametrize("kind", ["zero", "subnormal", "huge", "cancel"])
def test_gemv_edge_activations(V, kind):
    m = gen_matrix(1500, 2048, CONFIG0_PROBS, seed=30)
    x = _edge_x(m.K, kind, seed=31)
    y = _check_gemv(V, m, x)
    if kind == "zero":
        assert np.array_equal(y, np.zeros_like(y))


@pytest.mark.parametrize("kind", ["zero", "subnormal", "huge", "cancel"])
def test_smallbatch_edge_activations(V, kind):
    m = gen_matrix(1500, 2048, CONFIG0_PROBS, seed=32)
    X = np.stack([_edge_x(m.K, kind, seed=33 + j) for j in range(5)])
    mat = V.Matrix(m.codes, m.bits, m.scales)
    Y = gpu_gemm(V, mat, X)
    mat.close()
    ref = O.gemm(m.codes, m.bits, m.scales, X)
    PB.check_within(Y, ref, PB.tc_bound(m.codes, m.bits, m.scales, X))
    if kind == "zero":
        assert np.array_equal(Y, np.zeros_like(Y))


def test_smallbatch_all_rows_14336x4096_every_batch(V):
    m = gen_matrix(14336, 4096, CONFIG0_PROBS, seed=0)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    for B in (2, 3, 4, 8, 16, 32, 64):
        X = gen_x(m.K, seed=200 + B, batch=B)
        Y = gpu_gemm(V, mat, X)
        assert np.isfinite(Y).all(), B
        ref = O.gemm(m.codes, m.bits, m.scales, X)
        PB.check_within(Y, ref, PB.tc_bound(m.codes, m.bits, m.scales, X))
        assert gemv_err(m, X, Y) <= TOL, B
    mat.close()


@pytest.mark.parametrize("B", [65, 130, 200])
def test_gemm_prefill_batches(V, B):
    """vbq_gemm above 64 columns (blocks of 64 on the tensor cores, a short last block on the CUDA
    cores): every element within the tensor-core bound, which also covers the CUDA-core columns."""
    import torch
    m = gen_matrix(1500, 2048, CONFIG0_PROBS, seed=40)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    X = gen_x(m.K, seed=41 + B, batch=B)
    Y = torch.full((B, m.N), float("nan"), device="cuda")
    V.vbq_gemm(mat.handle, dev_u16(X), B, Y)
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    mat.close()
    assert np.isfinite(got).all()
    ref = O.gemm(m.codes, m.bits, m.scales, X)
    PB.check_within(got, ref, PB.tc_bound(m.codes, m.bits, m.scales, X))
    assert gemv_err(m, X, got) <= TOL
