"""ctypes binding to libvbq.so. Argument marshalling only; every step runs in the library.

The names follow the C ABI in include/vbq.h. Device pointers may be given as
ints or as torch tensors (their data_ptr()). Host arrays are numpy arrays.
stream=None means torch's current CUDA stream when torch is available, and the
legacy default stream otherwise. Errors raise VbqError with the library's status
and detail text.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libvbq.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "vbq.h")

VBQ_OK = 0
STATUS_NAMES = {0: "VBQ_OK", 1: "VBQ_ERR_INVALID_ARG", 2: "VBQ_ERR_SHAPE", 3: "VBQ_ERR_CODE_RANGE",
                4: "VBQ_ERR_BITS", 5: "VBQ_ERR_CUDA", 6: "VBQ_ERR_OOM", 7: "VBQ_ERR_DEVICE_CHECK",
                8: "VBQ_ERR_UNSUPPORTED"}


class VbqError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str):
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status
        self.detail = detail


class VbqInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("code_bytes", ctypes.c_int64),
                ("meta_bytes", ctypes.c_int64), ("total_bytes", ctypes.c_int64), ("mean_bits", ctypes.c_double),
                ("n_tiles", ctypes.c_int32), ("n_steps", ctypes.c_int32), ("groups_by_bits", ctypes.c_int64 * 4)]


class VbqModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_ST = ctypes.c_int


class VbqDenseJob(ctypes.Structure):
    """vbq_dense_job: device pointers and the shape of one dense GEMV."""
    _fields_ = [("W", _P), ("x", _P), ("y", _P), ("N", _I64), ("K", _I64)]


VBQ_DENSE_MAX_JOBS = 256


_SIGNATURES = {
    "vbq_status_str": (ctypes.c_char_p, [_ST]),
    "vbq_last_error": (ctypes.c_char_p, []),
    "vbq_pack": (_ST, [_P, _P, _P, _I64, _I64, _P, ctypes.POINTER(_P)]),
    "vbq_quantize_rtn": (_ST, [_P, _I64, _I64, _P, _P, _P]),
    "vbq_fakequant_forward": (_ST, [_P, _P, _P, ctypes.c_float, _I64, _I64, _P, _P]),
    "vbq_fakequant_backward": (_ST, [_P, _P, _P, ctypes.c_float, _P, _I64, _I64, _P, _P, _P]),
    "vbq_matrix_free": (None, [_P]),
    "vbq_matrix_info": (_ST, [_P, ctypes.POINTER(VbqInfo)]),
    "vbq_dequant": (_ST, [_P, _P, _P]),
    "vbq_gemv": (_ST, [_P, _P, _P, _P]),
    "vbq_gemm_smallbatch": (_ST, [_P, _P, _I32, _P, _P]),
    "vbq_gemm": (_ST, [_P, _P, _I64, _P, _P]),
    "vbq_model_create": (_ST, [ctypes.POINTER(VbqModelDesc), ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "vbq_model_free": (None, [_P]),
    "vbq_decode_step": (_ST, [_P, _P, _P, _P]),
    "vbq_decode_step_host": (_ST, [_P, _P, _P, _P]),
    "vbq_decode_step_noalloc": (_ST, [_P, _P, _P, _P]),
    "vbq_model_set_trace": (_ST, [_P, _I32]),
    "vbq_model_set_context": (_ST, [_P, _I32, ctypes.c_double]),
    "vbq_model_kv_cache": (_ST, [_P, _I32, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_I64)]),
    "vbq_decode_step_at": (_ST, [_P, _P, _I32, _P, _P]),
    "vbq_model_trace_info": (_ST, [_P, _P, _P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "vbq_model_read_trace": (_ST, [_P, _P, _P]),
    "vbq_dense_gemv_bf16": (_ST, [_P, _P, _P, _I64, _I64, _P]),
    "vbq_dense_gemv_bf16_many": (_ST, [_P, _I32, _P]),
    "vbq_rope_append": (_ST, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I64, _I32, ctypes.c_double, _P]),
    "vbq_attention_decode": (_ST, [_P, _P, _P, _I32, _I32, _I32, _I64, _I32, _P, _P]),
    "vbq_device_check": (_ST, [ctypes.POINTER(_I32)]),
    "vbq_launch_count": (_I64, [_I32]),
    "vbq_debug_set": (_ST, [_I32, _I64]),
}

_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libvbq.so; raises ImportError if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libvbq.so is not built ({path}); run: python mixed_precision_weight_bit_b300/build.py")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def _L() -> ctypes.CDLL:
    return _lib if _lib is not None else load_library()


def _check(func: str, status: int) -> None:
    if status != VBQ_OK:
        raise VbqError(func, status, _L().vbq_last_error().decode())


def _dptr(t) -> int:
    """Device pointer of a torch tensor or an int."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def vbq_status_str(status: int) -> str:
    return _L().vbq_status_str(status).decode()


def vbq_last_error() -> str:
    return _L().vbq_last_error().decode()


def vbq_pack(codes: np.ndarray, bits: np.ndarray, scales_f16: np.ndarray, stream=None) -> int:
    """Packs host arrays (codes u8 [N,K], bits u8 [N,K/64], scales u16 fp16 bits [N,K/64]); returns a handle."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    scales_f16 = np.ascontiguousarray(scales_f16, dtype=np.uint16)
    if codes.ndim != 2:
        raise ValueError("codes must be [N, K]")
    n, k = codes.shape
    out = _P()
    _check("vbq_pack", _L().vbq_pack(codes.ctypes.data, bits.ctypes.data, scales_f16.ctypes.data, n, k,
                                     _stream(stream), ctypes.byref(out)))
    return int(out.value)


def vbq_matrix_free(handle: int) -> None:
    _L().vbq_matrix_free(handle)


def vbq_matrix_info(handle: int) -> dict:
    info = VbqInfo()
    _check("vbq_matrix_info", _L().vbq_matrix_info(handle, ctypes.byref(info)))
    d = {f: getattr(info, f) for f, _ in VbqInfo._fields_ if f != "groups_by_bits"}
    d["groups_by_bits"] = {b: int(info.groups_by_bits[i]) for i, b in enumerate((1, 2, 4, 8))}
    return d


def vbq_dequant(handle: int, W, stream=None) -> None:
    _check("vbq_dequant", _L().vbq_dequant(handle, _dptr(W), _stream(stream)))


def vbq_fakequant_forward(W, alpha, u, tau: float, N: int, K: int, W_mix, stream=None) -> None:
    _check("vbq_fakequant_forward", _L().vbq_fakequant_forward(_dptr(W), _dptr(alpha), _dptr(u), float(tau), int(N),
                                                               int(K), _dptr(W_mix), _stream(stream)))


def vbq_fakequant_backward(W, alpha, u, tau: float, G, N: int, K: int, dW, dalpha, stream=None) -> None:
    _check("vbq_fakequant_backward", _L().vbq_fakequant_backward(_dptr(W), _dptr(alpha), _dptr(u), float(tau),
                                                                 _dptr(G), int(N), int(K), _dptr(dW), _dptr(dalpha),
                                                                 _stream(stream)))


def vbq_quantize_rtn(W: np.ndarray, bits: np.ndarray):
    """Dense float [N][K] weights at a bit map [N][K/64] -> (codes uint8 [N][K], scales fp16 bits [N][K/64])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    n, k = W.shape
    codes = np.zeros((n, k), np.uint8)
    scales = np.zeros((n, k // 64 if k % 64 == 0 else 0), np.uint16)
    _check("vbq_quantize_rtn", _L().vbq_quantize_rtn(W.ctypes.data, n, k, bits.ctypes.data, codes.ctypes.data,
                                                     scales.ctypes.data))
    return codes, scales


def vbq_gemv(handle: int, x, y, stream=None) -> None:
    _check("vbq_gemv", _L().vbq_gemv(handle, _dptr(x), _dptr(y), _stream(stream)))


def vbq_gemm_smallbatch(handle: int, X, B: int, Y, stream=None) -> None:
    _check("vbq_gemm_smallbatch", _L().vbq_gemm_smallbatch(handle, _dptr(X), int(B), _dptr(Y), _stream(stream)))


def vbq_gemm(handle: int, X, B: int, Y, stream=None) -> None:
    _check("vbq_gemm", _L().vbq_gemm(handle, _dptr(X), int(B), _dptr(Y), _stream(stream)))


def make_model_desc(n_layers, d, n_heads, n_kv_heads, head_dim, d_ff, vocab, rms_eps=1e-5) -> VbqModelDesc:
    return VbqModelDesc(n_layers, d, n_heads, n_kv_heads, head_dim, d_ff, vocab, rms_eps)


def vbq_model_create(desc: VbqModelDesc, mats: Sequence[int]) -> int:
    arr = (_P * len(mats))(*mats)
    out = _P()
    _check("vbq_model_create", _L().vbq_model_create(ctypes.byref(desc), arr, ctypes.byref(out)))
    return int(out.value)


def vbq_model_free(model: int) -> None:
    _L().vbq_model_free(model)


def vbq_decode_step(model: int, x, logits, stream=None) -> None:
    _check("vbq_decode_step", _L().vbq_decode_step(model, _dptr(x), _dptr(logits), _stream(stream)))


def vbq_decode_step_noalloc(model: int, x, logits, stream=None) -> None:
    _check("vbq_decode_step_noalloc",
           _L().vbq_decode_step_noalloc(model, _dptr(x), _dptr(logits), _stream(stream)))


def _hptr(a) -> int:
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("host array must be contiguous")
        return a.ctypes.data
    return int(a.data_ptr())  # pinned torch CPU tensor


def vbq_decode_step_host(model: int, x_host, logits_host, stream=None) -> None:
    _check("vbq_decode_step_host",
           _L().vbq_decode_step_host(model, _hptr(x_host), _hptr(logits_host), _stream(stream)))


def vbq_model_set_trace(model: int, enable: bool) -> None:
    _check("vbq_model_set_trace", _L().vbq_model_set_trace(model, 1 if enable else 0))


def vbq_model_trace_info(model: int, n_proj: int):
    in_off = np.zeros(n_proj, np.int64)
    out_off = np.zeros(n_proj, np.int64)
    it, ot = _I64(), _I64()
    _check("vbq_model_trace_info", _L().vbq_model_trace_info(model, in_off.ctypes.data, out_off.ctypes.data,
                                                             ctypes.byref(it), ctypes.byref(ot)))
    return in_off, out_off, int(it.value), int(ot.value)


def vbq_model_read_trace(model: int, in_total: int, out_total: int):
    tin = np.zeros(in_total, np.uint16)
    tout = np.zeros(out_total, np.float32)
    _check("vbq_model_read_trace", _L().vbq_model_read_trace(model, tin.ctypes.data, tout.ctypes.data))
    return tin, tout


def vbq_model_set_context(model: int, max_context: int, rope_theta: float = 10000.0) -> None:
    _check("vbq_model_set_context", _L().vbq_model_set_context(model, int(max_context), float(rope_theta)))


def vbq_model_kv_cache(model: int, layer: int):
    """(k_ptr, v_ptr, stride): device addresses of the layer's bf16 caches [n_kv_heads][stride][head_dim]."""
    k, v, st = _P(), _P(), _I64()
    _check("vbq_model_kv_cache", _L().vbq_model_kv_cache(model, int(layer), ctypes.byref(k), ctypes.byref(v),
                                                         ctypes.byref(st)))
    return int(k.value), int(v.value), int(st.value)


def vbq_decode_step_at(model: int, x, pos: int, logits, stream=None) -> None:
    _check("vbq_decode_step_at", _L().vbq_decode_step_at(model, _dptr(x), int(pos), _dptr(logits), _stream(stream)))


def vbq_dense_gemv_bf16(W, x, y, N: int, K: int, stream=None) -> None:
    _check("vbq_dense_gemv_bf16", _L().vbq_dense_gemv_bf16(_dptr(W), _dptr(x), _dptr(y), int(N), int(K),
                                                           _stream(stream)))


def vbq_dense_gemv_bf16_many(jobs, stream=None) -> None:
    """jobs: sequence of (W, x, y, N, K) with device tensors or pointers; one launch for all."""
    arr = (VbqDenseJob * max(1, len(jobs)))()
    for i, (W, x, y, N, K) in enumerate(jobs):
        arr[i] = VbqDenseJob(_dptr(W), _dptr(x), _dptr(y), int(N), int(K))
    _check("vbq_dense_gemv_bf16_many", _L().vbq_dense_gemv_bf16_many(ctypes.cast(arr, _P), len(jobs),
                                                                     _stream(stream)))


def vbq_rope_append(q, k_new, v_new, k_cache, v_cache, n_heads: int, n_kv_heads: int, head_dim: int,
                    kv_stride: int, pos: int, theta: float = 10000.0, stream=None) -> None:
    _check("vbq_rope_append", _L().vbq_rope_append(_dptr(q), _dptr(k_new), _dptr(v_new), _dptr(k_cache),
                                                   _dptr(v_cache), int(n_heads), int(n_kv_heads), int(head_dim),
                                                   int(kv_stride), int(pos), float(theta), _stream(stream)))


def vbq_attention_decode(q, k_cache, v_cache, n_heads: int, n_kv_heads: int, head_dim: int, kv_stride: int,
                         T: int, out, stream=None) -> None:
    _check("vbq_attention_decode", _L().vbq_attention_decode(_dptr(q), _dptr(k_cache), _dptr(v_cache), int(n_heads),
                                                             int(n_kv_heads), int(head_dim), int(kv_stride), int(T),
                                                             _dptr(out), _stream(stream)))


def vbq_device_check() -> int:
    """Returns the device check code (0 if clean); raises VbqError on a set code."""
    code = _I32()
    _check("vbq_device_check", _L().vbq_device_check(ctypes.byref(code)))
    return int(code.value)


def vbq_launch_count(reset: bool = False) -> int:
    return int(_L().vbq_launch_count(1 if reset else 0))


VBQ_DEBUG_WAIT_LIMIT = 1
VBQ_DEBUG_NEVER_READY = 2
VBQ_DEBUG_NOALLOC_WORDS = 3
VBQ_DEBUG_ALLOC_CAP = 4


def vbq_debug_set(key: int, value: int) -> None:
    """Test hooks of the decode step (see include/vbq.h); value 0 restores the default."""
    _check("vbq_debug_set", _L().vbq_debug_set(int(key), int(value)))


class Matrix:
    """Owns a packed matrix handle (freed by close() or garbage collection)."""

    def __init__(self, codes, bits, scales_f16, stream=None):
        self.handle = vbq_pack(codes, bits, scales_f16, stream)
        self.N, self.K = int(np.shape(codes)[0]), int(np.shape(codes)[1])

    def info(self) -> dict:
        return vbq_matrix_info(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", 0):
            vbq_matrix_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Model:
    """Owns a decode-step model over Matrix objects it keeps alive."""

    def __init__(self, desc: VbqModelDesc, mats: Sequence[Matrix]):
        self.mats = list(mats)
        self.desc = desc
        self.handle = vbq_model_create(desc, [m.handle for m in self.mats])

    def close(self) -> None:
        if getattr(self, "handle", 0):
            vbq_model_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
