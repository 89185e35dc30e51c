"""ctypes front end of the C++ oracle (oracle/vbq_oracle.cpp).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this module. ``build()`` compiles the
library with g++ into ``oracle/lib/`` (single-threaded, -O2, no fused
multiply-adds); the functions below take the same numpy arrays as
oracle/vbq_oracle.py and raise ValueError where it does.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Callable, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vbq_oracle.cpp")
LIB = os.path.join(HERE, "lib", "libvbq_oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle library if it is missing or older than its source; returns its path."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        os.makedirs(os.path.dirname(LIB), exist_ok=True)
        tmp = LIB + ".tmp"
        subprocess.run(["g++", *CXXFLAGS, "-o", tmp, SRC], check=True)
        os.replace(tmp, LIB)
    return LIB


class Model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_double)]


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        for name in ("vbq_oracle_dequant", "vbq_oracle_gemv", "vbq_oracle_row_norms"):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
        L.vbq_oracle_dequant.argtypes = [P, P, P, I64, I64, P]
        L.vbq_oracle_gemv.argtypes = [P, P, P, I64, I64, P, P]
        L.vbq_oracle_row_norms.argtypes = [P, P, P, I64, I64, P]
        L.vbq_oracle_to_bf16.argtypes = [P, I64, P]
        L.vbq_oracle_to_bf16.restype = None
        L.vbq_oracle_decode_step.argtypes = [ctypes.POINTER(Model), P, P, P, P, P]
        L.vbq_oracle_decode_step.restype = ctypes.c_int
        _lib = L
    return _lib


def _mat(codes, bits, scales):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    n, k = codes.shape
    if k % 64 or bits.shape != (n, k // 64) or scales.shape != (n, k // 64):
        raise ValueError("shapes: codes [N, K], bits and scales [N, K/64], K a multiple of 64")
    return codes, bits, scales, n, k


def dequant(codes, bits, scales) -> np.ndarray:
    codes, bits, scales, n, k = _mat(codes, bits, scales)
    W = np.empty((n, k), dtype=np.float32)
    if lib().vbq_oracle_dequant(codes.ctypes.data, bits.ctypes.data, scales.ctypes.data, n, k, W.ctypes.data):
        raise ValueError("invalid bit-width or code")
    return W


def gemv(codes, bits, scales, x_bits) -> np.ndarray:
    codes, bits, scales, n, k = _mat(codes, bits, scales)
    x = np.ascontiguousarray(np.asarray(x_bits).reshape(-1), dtype=np.uint16)
    if x.size != k:
        raise ValueError("x must have K entries")
    y = np.empty(n, dtype=np.float64)
    if lib().vbq_oracle_gemv(codes.ctypes.data, bits.ctypes.data, scales.ctypes.data, n, k, x.ctypes.data,
                             y.ctypes.data):
        raise ValueError("invalid bit-width or code")
    return y


def gemm(codes, bits, scales, X_bits) -> np.ndarray:
    X = np.asarray(X_bits)
    if X.ndim == 1:
        return gemv(codes, bits, scales, X)
    return np.stack([gemv(codes, bits, scales, X[j]) for j in range(X.shape[0])])


def row_norms(codes, bits, scales) -> np.ndarray:
    codes, bits, scales, n, k = _mat(codes, bits, scales)
    out = np.empty(n, dtype=np.float64)
    if lib().vbq_oracle_row_norms(codes.ctypes.data, bits.ctypes.data, scales.ctypes.data, n, k, out.ctypes.data):
        raise ValueError("invalid bit-width or code")
    return out


def to_bf16_bits(v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64).reshape(-1))
    out = np.empty(v.size, dtype=np.uint16)
    lib().vbq_oracle_to_bf16(v.ctypes.data, v.size, out.ctypes.data)
    return out


MatrixGetter = Callable[[int, str], Tuple[np.ndarray, np.ndarray, np.ndarray]]
PROJS = ("q", "k", "v", "o", "gate", "up", "down")


def decode_step(get_matrix: MatrixGetter, n_layers: int, n_heads: int, n_kv_heads: int, head_dim: int, d: int,
                d_ff: int, vocab: int, x_bits, eps: float = 1e-5) -> np.ndarray:
    """Logits of one decode step (the chain of oracle/vbq_oracle.py's decode_step), in C++."""
    keep = []
    for layer in range(n_layers):
        for p in PROJS:
            keep.append(_mat(*get_matrix(layer, p))[:3])
    keep.append(_mat(*get_matrix(n_layers, "head"))[:3])
    n = len(keep)
    C = (ctypes.c_void_p * n)(*[m[0].ctypes.data for m in keep])
    B = (ctypes.c_void_p * n)(*[m[1].ctypes.data for m in keep])
    S = (ctypes.c_void_p * n)(*[m[2].ctypes.data for m in keep])
    x = np.ascontiguousarray(np.asarray(x_bits).reshape(-1), dtype=np.uint16)
    desc = Model(n_layers, d, n_heads, n_kv_heads, head_dim, d_ff, vocab, eps)
    out = np.empty(vocab, dtype=np.float64)
    if lib().vbq_oracle_decode_step(ctypes.byref(desc), C, B, S, x.ctypes.data, out.ctypes.data):
        raise ValueError("invalid shapes or matrices")
    return out
