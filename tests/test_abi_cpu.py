"""The C-ABI library builds, loads and exports every declared symbol; host-side validation (CPU only)."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from tests.gpu_util import build_lib
    path = build_lib()
    from mixed_precision_weight_bit_b300 import vbq as V
    return V.load_library(path)


def declared_functions():
    with open(os.path.join(ROOT, "include", "vbq.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"VBQ_API\s+[\w\s\*]*?\b(vbq_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for must in ("vbq_pack", "vbq_dequant", "vbq_gemv", "vbq_gemm_smallbatch", "vbq_decode_step",
                 "vbq_model_create", "vbq_matrix_info", "vbq_status_str"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol(lib):
    from mixed_precision_weight_bit_b300 import vbq as V
    for name in declared_functions():
        assert name in V._SIGNATURES, name
        assert callable(getattr(V, name)), name


def test_status_strings(lib):
    from mixed_precision_weight_bit_b300 import vbq as V
    for code, name in V.STATUS_NAMES.items():
        assert V.vbq_status_str(code) == name


def test_pack_validation_errors_without_gpu(lib):
    """Every check below fails before any CUDA call, so it runs on a CPU-only host."""
    from mixed_precision_weight_bit_b300 import vbq as V
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 2, size=(4, 128)).astype(np.uint8)
    bits = np.ones((4, 2), np.uint8)
    scales = np.full((4, 2), 0x3C00, np.uint16)
    with pytest.raises(V.VbqError) as e:
        V.vbq_pack(codes[:, :100], np.ones((4, 2), np.uint8), scales)
    assert e.value.status == 2  # K % 64
    bad = bits.copy()
    bad[1, 1] = 3
    with pytest.raises(V.VbqError) as e:
        V.vbq_pack(codes, bad, scales)
    assert e.value.status == 4 and "group index 3" in e.value.detail
    badc = codes.copy()
    badc[2, 70] = 2  # 1-bit group holding code 2
    with pytest.raises(V.VbqError) as e:
        V.vbq_pack(badc, bits, scales)
    assert e.value.status == 3
    out = ctypes.c_void_p()
    st = lib.vbq_pack(None, None, None, 4, 128, None, ctypes.byref(out))
    assert st == 1 and out.value is None
    assert lib.vbq_pack(None, None, None, -1, 64, None, ctypes.byref(out)) == 2
    assert lib.vbq_pack(None, None, None, 1, 64 * 65536, None, ctypes.byref(out)) == 2


def test_null_handles_rejected(lib):
    from mixed_precision_weight_bit_b300 import vbq as V
    for fn, args in (("vbq_gemv", (None, None, None, None)), ("vbq_dequant", (None, None, None)),
                     ("vbq_gemm_smallbatch", (None, None, 1, None, None)),
                     ("vbq_decode_step", (None, None, None, None))):
        assert getattr(lib, fn)(*args) == 1, fn
    assert lib.vbq_model_create(None, None, None) == 1
    info = V.VbqInfo()
    assert lib.vbq_matrix_info(None, ctypes.byref(info)) == 1


def test_dense_many_validation_without_gpu(lib):
    """The batched dense baseline checks every job before it launches anything."""
    from mixed_precision_weight_bit_b300 import vbq as V
    with pytest.raises(V.VbqError) as e:
        V.vbq_dense_gemv_bf16_many([(None, None, None, 4, 8)] * (V.VBQ_DENSE_MAX_JOBS + 1))
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_dense_gemv_bf16_many([(16, 16, 16, 4, 12)])   # K % 8
    assert e.value.status == 2
    with pytest.raises(V.VbqError) as e:
        V.vbq_dense_gemv_bf16_many([(16, 16, None, 4, 8)])  # NULL y
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_dense_gemv_bf16_many([(16, 16, 16, 4, 8), (18, 16, 16, 4, 8)])  # W not 16-byte aligned
    assert e.value.status == 1
    assert lib.vbq_dense_gemv_bf16_many(None, 1, None) == 1


def test_attention_validation_without_gpu(lib):
    """Shape and argument checks of the attention calls come before any CUDA call."""
    from mixed_precision_weight_bit_b300 import vbq as V
    p = 1 << 20  # a 16-byte aligned stand-in address; nothing is launched
    bad = [
        dict(n_heads=32, n_kv_heads=8, head_dim=96, kv_stride=16, T=4),     # head_dim
        dict(n_heads=30, n_kv_heads=8, head_dim=128, kv_stride=16, T=4),    # H % H_kv
        dict(n_heads=72, n_kv_heads=8, head_dim=128, kv_stride=16, T=4),    # 9 query heads per kv head
        dict(n_heads=32, n_kv_heads=8, head_dim=128, kv_stride=16, T=0),    # T
        dict(n_heads=32, n_kv_heads=8, head_dim=128, kv_stride=16, T=17),   # T > kv_stride
        dict(n_heads=32, n_kv_heads=8, head_dim=128, kv_stride=70000, T=65537),
    ]
    for kw in bad:
        with pytest.raises(V.VbqError) as e:
            V.vbq_attention_decode(p, p, p, kw["n_heads"], kw["n_kv_heads"], kw["head_dim"], kw["kv_stride"],
                                   kw["T"], p)
        assert e.value.status == 2, kw
    with pytest.raises(V.VbqError) as e:
        V.vbq_attention_decode(p, None, p, 32, 8, 128, 16, 4, p)
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_attention_decode(p, p + 2, p, 32, 8, 128, 16, 4, p)   # cache not 16-byte aligned
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_rope_append(p, p, p, p, p, 32, 8, 128, 16, 16)         # pos >= kv_stride
    assert e.value.status == 2
    with pytest.raises(V.VbqError) as e:
        V.vbq_rope_append(p, p, p, p, p, 32, 8, 128, 16, 3, theta=1.0)
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_rope_append(p, p, None, p, p, 32, 8, 128, 16, 3)
    assert e.value.status == 1


def test_gemm_validation_without_gpu(lib):
    assert lib.vbq_gemm(None, None, 65, None, None) == 1
    from mixed_precision_weight_bit_b300 import vbq as V
    with pytest.raises(V.VbqError) as e:
        V.vbq_gemm(0, 0, 128, 0)
    assert e.value.status == 1


def test_fakequant_validation_without_gpu(lib):
    from mixed_precision_weight_bit_b300 import vbq as V
    p = 1 << 20
    with pytest.raises(V.VbqError) as e:
        V.vbq_fakequant_forward(p, p, p, 1.0, 4, 100, p)      # K % 64
    assert e.value.status == 2
    with pytest.raises(V.VbqError) as e:
        V.vbq_fakequant_forward(p, p, p, 0.0, 4, 64, p)       # tau
    assert e.value.status == 1
    with pytest.raises(V.VbqError) as e:
        V.vbq_fakequant_backward(p, p, p, 1.0, None, 4, 64, p, p)
    assert e.value.status == 1
    # 16-byte pieces: W, W_mix, G and dW must be 16-byte aligned; 8 is not enough
    for args in [(p + 8, p, p, 1.0, 4, 64, p), (p, p, p, 1.0, 4, 64, p + 8)]:
        with pytest.raises(V.VbqError) as e:
            V.vbq_fakequant_forward(*args)
        assert e.value.status == 1 and "align" in str(e.value)
    for args in [(p, p, p, 1.0, p + 8, 4, 64, p, p), (p, p, p, 1.0, p, 4, 64, p + 8, p)]:
        with pytest.raises(V.VbqError) as e:
            V.vbq_fakequant_backward(*args)
        assert e.value.status == 1 and "align" in str(e.value)

