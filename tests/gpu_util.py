"""Helpers for the GPU parity tests: run the library through the C ABI, compare with the oracle."""

from __future__ import annotations

import numpy as np

from oracle import vbq_oracle as O

TOL = 2e-3  # max |y - y_ref| / (||W_r|| ||x||), the parity bar for every GEMV/GEMM


def build_lib() -> str:
    """Builds libvbq.so in-tree (no-op when up to date) and returns its path.

    The build script is loaded by path, since importing the package loads the
    library and fails while it is missing.
    """
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location(
        "_vbq_build", os.path.join(root, "mixed_precision_weight_bit_b300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def lib():
    build_lib()
    import mixed_precision_weight_bit_b300 as V
    return V


def dev_u16(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def gpu_gemv(V, mat, x: np.ndarray) -> np.ndarray:
    import torch
    y = torch.full((mat.N,), float("nan"), dtype=torch.float32, device="cuda")
    V.vbq_gemv(mat.handle, dev_u16(x), y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def gpu_gemm(V, mat, X: np.ndarray) -> np.ndarray:
    import torch
    B = X.shape[0]
    Y = torch.full((B, mat.N), float("nan"), dtype=torch.float32, device="cuda")
    V.vbq_gemm_smallbatch(mat.handle, dev_u16(X), B, Y)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


def gpu_dequant(V, mat) -> np.ndarray:
    import torch
    W = torch.full((mat.N, mat.K), float("nan"), dtype=torch.float32, device="cuda")
    V.vbq_dequant(mat.handle, W)
    torch.cuda.synchronize()
    return W.cpu().numpy()


def gemv_err(m, x, y_gpu, rows=None) -> float:
    codes, bits, scales = m.codes, m.bits, m.scales
    if rows is not None:
        codes, bits, scales, y_gpu = codes[rows], bits[rows], scales[rows], y_gpu[..., rows]
    y_ref = O.gemm(codes, bits, scales, x)
    return O.normalized_error(y_gpu, y_ref, O.row_norms(codes, bits, scales), x)


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two bf16 arrays of the same sign convention."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, 0x8000 - (a & 0x7FFF), 0x8000 + a)
    b = np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(a - b)
