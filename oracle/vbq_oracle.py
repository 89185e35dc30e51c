"""CPU oracle for the VBQ decode path: plain, slow and written to be checked by eye.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this module. The library never calls it,
and it shares no code with the CUDA path.

What it follows:

* "Variable Bit-width Quantization: Learning Per-Group Precision for
  'Bigger-but-Smaller' Language Models", abstract. Every run of 64 consecutive
  weights gets its own bit-width from {1,2,4,8}; the learned allocation is
  stored as packed low-bit codes, and kernels that dequantize inside the
  multiply speed up token-by-token decode. The abstract gives no code grid, so the
  grid is the one this project fixes: w = s_g * (q - (2^b_g - 1)/2). Here s_g is
  an fp16 scale and q is an unsigned code in [0, 2^b_g - 1]. Group g of row r
  covers columns [64g, 64g + 63].
* The projections of one decode step follow the same abstract (token-by-token
  decode). The pages give no architecture, so the glue between projections is
  this project's reading:
  - unit-gamma RMSNorm with eps 1e-5;
  - attention at position 0, where a softmax over one key is 1, so each head
    outputs its kv-group's v;
  - SwiGLU, and residual adds;
  - bf16 rounding (round to nearest, ties to even) of every projection input.

Precision: dequantization is done in fp32. It is exact: an fp16 scale has 11
significant bits, and q - c_b is a half-integer with at most 9, so the product
fits fp32's 24 bits. Dot products are done in fp64 on the exact fp32 weights and
the exact bf16 inputs.

Parity pins: see tests/test_oracle_pins.py. Every function in this module is
pinned by brute force in exact rational arithmetic, by a closed form, or by an
invariant.
"""

from __future__ import annotations

from typing import Callable, Dict, Optional, Tuple

import numpy as np

GROUP = 64
RMS_EPS = 1e-5


# --------------------------------------------------------------------------
# bf16 / fp16 value conversions
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (the upper half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round real values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits and fp32's exponent range. For
    v = m * 2^e with 0.5 <= |m| < 1 the last kept bit has weight 2^(e-8). Below
    the smallest normal (2^-126) the quantum stays at 2^-133. np.round rounds
    half to even, and dividing by a power of two is exact.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    out = np.round(v / quantum) * quantum
    return np.where(v == 0.0, v, out)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of bf16_round(v) (finite inputs)."""
    r = bf16_round(v).astype(np.float32)  # exact: a bf16 value is an fp32 value
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# The code grid and dequantization
# --------------------------------------------------------------------------

def grid_offset(bits: np.ndarray) -> np.ndarray:
    """c_b = (2^b - 1) / 2 for each group's bit-width b (exact in fp32)."""
    b = np.asarray(bits, dtype=np.int64)
    return ((np.left_shift(1, b) - 1).astype(np.float64) / 2.0).astype(np.float32)


def check_inputs(codes: np.ndarray, bits: np.ndarray, scales: np.ndarray) -> Tuple[int, int, int]:
    n, k = codes.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of 64")
    g = k // GROUP
    if bits.shape != (n, g) or scales.shape != (n, g):
        raise ValueError("bits/scales must be [N, K/64]")
    if not np.isin(bits, (1, 2, 4, 8)).all():
        raise ValueError("bit-widths must be in {1,2,4,8}")
    lim = (np.left_shift(1, bits.astype(np.int64)) - 1)
    if (codes.reshape(n, g, GROUP).astype(np.int64) > lim[:, :, None]).any():
        raise ValueError("code out of range for its group's bit-width")
    return n, k, g


def dequant(codes: np.ndarray, bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[r, k] = s_{r,g} * (q_{r,k} - c_{b_{r,g}}), g = k // 64, in fp32 (exact)."""
    n, k, g = check_inputs(codes, bits, scales)
    s = np.asarray(scales, dtype=np.uint16).view(np.float16).astype(np.float32)
    c = grid_offset(bits)
    q = codes.reshape(n, g, GROUP).astype(np.float32)
    w = s[:, :, None] * (q - c[:, :, None])
    return w.reshape(n, k)


def _row_chunks(n: int, k: int, budget_bytes: int = 256 << 20):
    rows = max(1, budget_bytes // max(1, 8 * k))
    for r0 in range(0, n, rows):
        yield r0, min(n, r0 + rows)


def gemm(codes: np.ndarray, bits: np.ndarray, scales: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """Y[j, r] = sum_k W[r, k] * X[j, k] in fp64, for bf16 X [B, K] (or x [K])."""
    x = bf16_bits_to_f64(x_bits)
    squeeze = x.ndim == 1
    X = x[None, :] if squeeze else x
    n, k = codes.shape
    Y = np.empty((X.shape[0], n), dtype=np.float64)
    for r0, r1 in _row_chunks(n, k):
        W = dequant(codes[r0:r1], bits[r0:r1], scales[r0:r1]).astype(np.float64)
        Y[:, r0:r1] = X @ W.T
    return Y[0] if squeeze else Y


def gemv(codes: np.ndarray, bits: np.ndarray, scales: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """y = W x in fp64 for one bf16 activation vector."""
    return gemm(codes, bits, scales, np.asarray(x_bits).reshape(-1))


def row_norms(codes: np.ndarray, bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """||W_r||_2 of the dequantized rows (fp64)."""
    n, k = codes.shape
    out = np.empty(n, dtype=np.float64)
    for r0, r1 in _row_chunks(n, k):
        W = dequant(codes[r0:r1], bits[r0:r1], scales[r0:r1]).astype(np.float64)
        out[r0:r1] = np.sqrt((W * W).sum(axis=1))
    return out


def normalized_error(y_test: np.ndarray, y_ref: np.ndarray, w_row_norms: np.ndarray,
                     x_bits: np.ndarray) -> float:
    """max_r |y_test[r] - y_ref[r]| / (||W_r||_2 * ||x||_2) (max over batch columns too)."""
    x = bf16_bits_to_f64(x_bits)
    xn = np.sqrt((x * x).sum(axis=-1))
    yt = np.asarray(y_test, dtype=np.float64)
    yr = np.asarray(y_ref, dtype=np.float64)
    if yr.ndim == 1:
        denom = w_row_norms * xn
    else:
        denom = w_row_norms[None, :] * xn[:, None]
    denom = np.where(denom == 0.0, 1.0, denom)
    if yr.size == 0:
        return 0.0
    return float(np.max(np.abs(yt - yr) / denom))


def storage_bytes(bits: np.ndarray) -> Dict[str, float]:
    """Code bytes = sum over groups of 64 * b / 8; mean bits = 8 * code bytes / weights."""
    b = np.asarray(bits, dtype=np.int64)
    code_bytes = int((GROUP * b // 8).sum())
    weights = b.size * GROUP
    return {"code_bytes": code_bytes, "weights": weights,
            "mean_bits": 8.0 * code_bytes / weights if weights else 0.0}


# --------------------------------------------------------------------------
# Decode step (one token, position 0) through a stack of VBQ projections
# --------------------------------------------------------------------------

def rmsnorm(h: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps), unit gain, fp64."""
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h) + eps)


def silu(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def attention_pos0(v: np.ndarray, n_heads: int, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Attention output of one query over a single cached key (position 0).

    The softmax over one score is exactly 1, so query head i returns the value
    vector of its kv head i // (n_heads / n_kv_heads) (grouped-query attention).
    RoPE at position 0 is the identity, so q and k do not enter the result.
    """
    group = n_heads // n_kv_heads
    v = np.asarray(v, dtype=np.float64).reshape(n_kv_heads, head_dim)
    return np.concatenate([v[i // group] for i in range(n_heads)])


MatrixGetter = Callable[[int, str], Tuple[np.ndarray, np.ndarray, np.ndarray]]


AttendFn = Callable[[int, np.ndarray, np.ndarray, np.ndarray], np.ndarray]


def decode_step(get_matrix: MatrixGetter, n_layers: int, n_heads: int, n_kv_heads: int,
                head_dim: int, x_bits: np.ndarray, eps: float = RMS_EPS,
                trace: Optional[list] = None, attend: Optional[AttendFn] = None,
                dense: Optional[Callable[[int, str], np.ndarray]] = None) -> np.ndarray:
    """Logits of one decode step, fp64 throughout, bf16 at every projection input.

    get_matrix(layer, proj) returns (codes, bits, scales). proj is one of
    q, k, v, o, gate, up, down, and 'head' for layer n_layers.

    h <- x
    per layer: u = bf16(rmsnorm(h)); q, k, v = Wq u, Wk u, Wv u
               a = bf16(attention_pos0(v)); h <- h + Wo a
               u = bf16(rmsnorm(h)); m = bf16(silu(Wgate u) * (Wup u)); h <- h + Wdown m
    logits = Whead bf16(rmsnorm(h))

    If trace is a list, one (layer, proj, input_bits, output) tuple is appended per projection.
    attend(layer, q, k, v), if given, replaces attention_pos0 (a step at a later
    position: see oracle/attention_oracle.py); it returns the fp64 attention
    output [n_heads * head_dim], which is rounded to bf16 like every projection input.
    dense(layer, proj), if given, returns a dense weight matrix [N][K] used in
    place of get_matrix's packed one (the same chain over dense weights).
    """
    def proj(layer: int, name: str, inp_bits: np.ndarray) -> np.ndarray:
        if dense is not None:
            y = np.asarray(dense(layer, name), dtype=np.float64) @ bf16_bits_to_f64(inp_bits)
        else:
            y = gemv(*get_matrix(layer, name), inp_bits)
        if trace is not None:
            trace.append((layer, name, inp_bits.copy(), y))
        return y

    h = bf16_bits_to_f64(x_bits)
    for layer in range(n_layers):
        u = f64_to_bf16_bits(rmsnorm(h, eps))
        q = proj(layer, "q", u)
        k = proj(layer, "k", u)
        v = proj(layer, "v", u)
        att = attention_pos0(v, n_heads, n_kv_heads, head_dim) if attend is None else attend(layer, q, k, v)
        a = f64_to_bf16_bits(att)
        h = h + proj(layer, "o", a)
        u = f64_to_bf16_bits(rmsnorm(h, eps))
        g = proj(layer, "gate", u)
        up = proj(layer, "up", u)
        m = f64_to_bf16_bits(silu(g) * up)
        h = h + proj(layer, "down", m)
    u = f64_to_bf16_bits(rmsnorm(h, eps))
    return proj(n_layers, "head", u)
