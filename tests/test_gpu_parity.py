"""GPU parity of dequant / GEMV / small-batch GEMM against the CPU oracle, through the C ABI."""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import (CONFIG0_PROBS, bf16_bits_to_f32, gen_matrix, gen_matrix_with_bits, gen_stress, gen_x, stress_bits)
from tests.gpu_util import TOL, dev_u16, gemv_err, gpu_dequant, gpu_gemm, gpu_gemv, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _one_class(n, k, b, seed):
    return gen_matrix_with_bits(np.full((n, k // 64), b, np.uint8), seed, (8, b))


CASES = {
    "config0_768": lambda: gen_matrix(768, 768, CONFIG0_PROBS, seed=0),
    "ragged_1x64": lambda: gen_matrix(1, 64, CONFIG0_PROBS, seed=1),
    "ragged_3x128": lambda: gen_matrix(3, 128, CONFIG0_PROBS, seed=2),
    "ragged_300x1024": lambda: gen_matrix(300, 1024, CONFIG0_PROBS, seed=3),
    "ragged_257x640": lambda: gen_matrix(257, 640, CONFIG0_PROBS, seed=4),
    "ragged_511x192": lambda: gen_matrix(511, 192, CONFIG0_PROBS, seed=5),
    "tall_4099x128": lambda: gen_matrix(4099, 128, CONFIG0_PROBS, seed=6),
    "all1_200x512": lambda: _one_class(200, 512, 1, 7),
    "all2_200x512": lambda: _one_class(200, 512, 2, 8),
    "all4_200x512": lambda: _one_class(200, 512, 4, 9),
    "all8_200x512": lambda: _one_class(200, 512, 8, 10),
    "stress_a_1024": lambda: gen_stress("a", 1024, 1024),
    "stress_b_1024": lambda: gen_stress("b", 1024, 1024),
    "stress_c_1024": lambda: gen_stress("c", 1024, 1024),
    "stress_d_1024": lambda: gen_stress("d", 1024, 1024),
    "stress_e_1024": lambda: gen_stress("e", 1024, 1024),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_dequant_bit_exact(V, name):
    m = CASES[name]()
    mat = V.Matrix(m.codes, m.bits, m.scales)
    W = gpu_dequant(V, mat)
    ref = O.dequant(m.codes, m.bits, m.scales)
    assert np.array_equal(W.view(np.uint32), ref.view(np.uint32))
    mat.close()


@pytest.mark.parametrize("name", sorted(CASES))
def test_gemv_parity(V, name):
    m = CASES[name]()
    x = gen_x(m.K, seed=11)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    y = gpu_gemv(V, mat, x)
    assert np.isfinite(y).all()
    assert gemv_err(m, x, y) <= TOL
    mat.close()


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 7, 8, 9, 13, 16])
def test_smallbatch_parity(V, B):
    m = gen_matrix(300, 1024, CONFIG0_PROBS, seed=12)
    X = gen_x(m.K, seed=13, batch=B)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    Y = gpu_gemm(V, mat, X)
    assert np.isfinite(Y).all()
    assert gemv_err(m, X, Y) <= TOL
    # column j equals the batch-1 result on x_j up to summation order
    y0 = gpu_gemv(V, mat, X[0])
    assert gemv_err(m, X[0], y0) <= TOL
    mat.close()


def test_smallbatch_full_width(V):
    m = gen_matrix(1024, 4096, CONFIG0_PROBS, seed=14)
    X = gen_x(m.K, seed=15, batch=64)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    Y = gpu_gemm(V, mat, X)
    rows = np.r_[0:16, 1000:1024]
    assert gemv_err(m, X, Y, rows) <= TOL
    mat.close()


def test_deterministic(V):
    m = gen_matrix(2048, 2048, CONFIG0_PROBS, seed=16)
    x = gen_x(m.K, seed=17)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    a = gpu_gemv(V, mat, x)
    b = gpu_gemv(V, mat, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    mat.close()


def test_empty_shapes(V):
    import torch
    m0 = gen_matrix(0, 128, CONFIG0_PROBS, seed=18)
    mat = V.Matrix(m0.codes, m0.bits, m0.scales)
    assert mat.info()["n_tiles"] == 0
    V.vbq_gemv(mat.handle, dev_u16(gen_x(128, seed=1)), torch.empty(1, device="cuda"))
    mat.close()
    codes = np.zeros((5, 0), np.uint8)
    mat = V.Matrix(codes, np.zeros((5, 0), np.uint8), np.zeros((5, 0), np.uint16))
    y = torch.full((5,), 7.0, device="cuda")
    V.vbq_gemv(mat.handle, dev_u16(np.zeros(2, np.uint16)), y)
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    mat.close()


def test_misaligned_x_rejected(V):
    import torch
    m = gen_matrix(8, 128, CONFIG0_PROBS, seed=19)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    xb = torch.zeros(130, dtype=torch.int16, device="cuda")
    y = torch.zeros(8, device="cuda")
    with pytest.raises(V.VbqError) as e:
        V.vbq_gemv(mat.handle, xb.data_ptr() + 2, y)
    assert e.value.status == 1
    mat.close()


def test_info_accounting(V):
    m = gen_matrix(777, 1280, CONFIG0_PROBS, seed=20)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    info = mat.info()
    st = O.storage_bytes(m.bits)
    assert info["code_bytes"] == st["code_bytes"]
    assert info["mean_bits"] == pytest.approx(st["mean_bits"])
    assert info["total_bytes"] == info["code_bytes"] + info["meta_bytes"]
    for b in (1, 2, 4, 8):
        assert info["groups_by_bits"][b] == int((m.bits == b).sum())
    mat.close()


# ---- full sizes: sampled rows against the oracle ----

def _sample_rows(n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.r_[0, 1, n - 2, n - 1, rng.integers(0, n, 60)])


def test_full_14336x4096_batch_sweep(V):
    m = gen_matrix(14336, 4096, CONFIG0_PROBS, seed=0)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    rows = _sample_rows(m.N, 1)
    for B in (1, 2, 4, 8, 16, 32, 64):
        X = gen_x(m.K, seed=100 + B, batch=B)
        Y = gpu_gemm(V, mat, X)
        assert np.isfinite(Y).all()
        assert gemv_err(m, X, Y, rows) <= TOL, B
    mat.close()


@pytest.mark.parametrize("case", ["a", "b", "c", "d", "e"])
def test_full_stress_8192(V, case):
    m = gen_stress(case, 8192, 8192)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    x = gen_x(m.K, seed=21)
    y = gpu_gemv(V, mat, x)
    assert np.isfinite(y).all()
    assert gemv_err(m, x, y, _sample_rows(m.N, 2)) <= TOL
    mat.close()


def test_device_check_clean(V):
    assert V.vbq_device_check() == 0


# ---- batches of 16..64: the tensor-core dequant-MMA ----

TC_CASES = {
    "mix300x1024": lambda: gen_matrix(300, 1024, CONFIG0_PROBS, seed=30),      # tiles of < 256 rows, both halves
    "mix100x512": lambda: gen_matrix(100, 512, CONFIG0_PROBS, seed=31),        # one tile of <= 128 rows
    "mix777x64": lambda: gen_matrix(777, 64, CONFIG0_PROBS, seed=32),          # one group per row
    "all8_256x512": lambda: _one_class(256, 512, 8, 33),                       # the largest column span
    "all1_512x256": lambda: _one_class(512, 256, 1, 34),
    "stress_e_1024": lambda: gen_stress("e", 1024, 1024),
}


@pytest.mark.parametrize("name", sorted(TC_CASES))
@pytest.mark.parametrize("B", [16, 17, 31, 48, 64])
def test_tensor_core_batches(V, name, B):
    m = TC_CASES[name]()
    X = gen_x(m.K, seed=40 + B, batch=B)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    V.vbq_launch_count(reset=True)
    Y = gpu_gemm(V, mat, X)
    assert V.vbq_launch_count() == 3  # x scales, the B tiles, and one tensor-core launch for all B columns
    assert np.isfinite(Y).all()
    assert gemv_err(m, X, Y) <= TOL
    mat.close()
    assert V.vbq_device_check() == 0


def test_tensor_core_large_x_and_repeat(V):
    """x far outside fp16's range is scaled by a power of two per column; two calls agree bit for bit."""
    m = gen_matrix(512, 1024, CONFIG0_PROBS, seed=35)
    X = gen_x(m.K, seed=36, batch=24)
    Xf = bf16_bits_to_f32(X) * np.float32(2.0 ** 40)
    Xf[3] *= np.float32(2.0 ** -80)            # one column tiny
    from synth import f32_to_bf16_bits
    X = f32_to_bf16_bits(Xf)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    Y1 = gpu_gemm(V, mat, X)
    Y2 = gpu_gemm(V, mat, X)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    assert gemv_err(m, X, Y1) <= TOL
    mat.close()


def test_large_scales_take_the_cuda_core_path(V):
    """Scales whose products would overflow fp16 are served by the CUDA-core kernel, still within tolerance."""
    m = gen_matrix(200, 512, CONFIG0_PROBS, seed=37)
    scales = np.full_like(m.scales, np.float16(1000.0).view(np.uint16))
    X = gen_x(m.K, seed=38, batch=20)
    mat = V.Matrix(m.codes, m.bits, scales)
    Y = gpu_gemm(V, mat, X)
    from synth import VbqMatrixInputs
    ref = VbqMatrixInputs(codes=m.codes, bits=m.bits, scales=scales)
    assert gemv_err(ref, X, Y) <= TOL
    mat.close()


# ---- the dense bf16 baseline ----

@pytest.mark.parametrize("N,K", [(1, 8), (3, 72), (300, 1024), (4099, 4096)])
def test_dense_bf16_gemv(V, N, K):
    """y = W x for bf16 W and x with fp32 accumulation, against the fp64 product of the same bf16 values."""
    import torch
    rng = np.random.default_rng(N * 7919 + K)
    w_bits = O.f64_to_bf16_bits(rng.standard_normal((N, K)) * 0.05)
    x_bits = gen_x(K, seed=N + K)
    y = torch.full((N,), float("nan"), device="cuda")
    V.vbq_dense_gemv_bf16(dev_u16(w_bits), dev_u16(x_bits), y, N, K)
    torch.cuda.synchronize()
    w = O.bf16_bits_to_f64(w_bits)
    x = O.bf16_bits_to_f64(x_bits)
    ref = w @ x
    got = y.cpu().numpy().astype(np.float64)
    norms = np.linalg.norm(w, axis=1) * np.linalg.norm(x)
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - ref) / norms) <= TOL


def test_dense_bf16_gemv_many(V):
    """One launch for several dense GEMVs of different shapes (and an empty and a K = 0 job)."""
    import torch
    shapes = [(300, 1024), (0, 64), (7, 0), (4099, 4096), (1, 8), (1024, 14336), (65, 72)]
    jobs, refs = [], []
    for i, (N, K) in enumerate(shapes):
        rng = np.random.default_rng(1000 + i)
        w_bits = O.f64_to_bf16_bits(rng.standard_normal((N, K)) * 0.05)
        x_bits = gen_x(K, seed=2000 + i) if K else np.zeros(0, np.uint16)
        W = dev_u16(w_bits) if N * K else torch.empty(8, dtype=torch.int16, device="cuda")
        x = dev_u16(x_bits) if K else torch.empty(8, dtype=torch.int16, device="cuda")
        y = torch.full((max(N, 1),), float("nan"), device="cuda")
        jobs.append((W, x, y, N, K))
        w = O.bf16_bits_to_f64(w_bits).reshape(N, K)
        xf = O.bf16_bits_to_f64(x_bits)
        refs.append((w @ xf if N else np.zeros(0), np.linalg.norm(w, axis=1) * np.linalg.norm(xf)))
    V.vbq_dense_gemv_bf16_many(jobs)
    torch.cuda.synchronize()
    for (W, x, y, N, K), (ref, norms) in zip(jobs, refs):
        got = y.cpu().numpy()[:N].astype(np.float64)
        assert np.isfinite(got).all(), (N, K)
        if K == 0:
            assert np.array_equal(got, np.zeros(N))
        elif N:
            assert np.max(np.abs(got - ref) / norms) <= TOL, (N, K)

