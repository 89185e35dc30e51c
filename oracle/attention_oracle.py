"""CPU oracle for decode attention over a KV cache: plain fp64 numpy.

TEST INFRASTRUCTURE ONLY. Only the tests and the bench's CPU-baseline leg may
import this module. The library never calls it, and it shares no code with
the CUDA path.

The source pages say only that VBQ speeds up token-by-token ("autoregressive")
decode ("Variable Bit-width Quantization: Learning Per-Group Precision for
'Bigger-but-Smaller' Language Models", abstract); a decode step at context
above one also attends over the cached keys and values. The pages give no
attention variant, so this module writes out the standard definitions, as
this project reads them:

* rotary position embedding with the rotate-half pairing: for i < d/2 the pair
  (x_i, x_{i+d/2}) turns by the angle pos * theta^(-2i/d); the result is
  rounded to fp32 and then to bf16 (nearest even), as the cache stores bf16;
* scaled dot-product attention for one query token: for query head h and its
  kv head g = h // (H / H_kv), p = softmax_j(q_h . k_g[j] / sqrt(d)) over
  j < T, and out_h = sum_j p_j v_g[j].

Parity pins: tests/test_attention_oracle.py (identity at position 0, the
rotation's norm and composition, a hand case, T = 1, uniform and one-hot
scores, the grouping of query heads, and invariance under a permutation of
the positions).
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

from oracle.vbq_oracle import bf16_bits_to_f64, f64_to_bf16_bits


def rope_f64(x: np.ndarray, pos: int, theta: float = 10000.0) -> np.ndarray:
    """Rotary embedding of the rows of x ([n, d], fp64) at position pos, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * np.power(float(theta), -2.0 * i / d)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., :half], x[..., half:]
    return np.concatenate([x0 * c - x1 * s, x0 * s + x1 * c], axis=-1)


def rope_bf16(x_bits: np.ndarray, pos: int, theta: float = 10000.0) -> np.ndarray:
    """Rotary embedding of bf16 rows: fp64 rotation, rounded to fp32, then to bf16."""
    y = rope_f64(bf16_bits_to_f64(x_bits), pos, theta)
    return f64_to_bf16_bits(y.astype(np.float32).astype(np.float64))


def attention_decode(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, T: int
                     ) -> Tuple[np.ndarray, np.ndarray]:
    """One query token over positions j < T.

    q_bits: bf16 [H, d]; k_bits, v_bits: bf16 [H_kv, >= T, d].
    Returns (out [H, d] fp64, p [H, T] fp64 softmax weights).
    """
    q = bf16_bits_to_f64(q_bits)
    K = bf16_bits_to_f64(k_bits)[:, :T, :]
    V = bf16_bits_to_f64(v_bits)[:, :T, :]
    H, d = q.shape
    Hkv = K.shape[0]
    group = H // Hkv
    out = np.zeros((H, d))
    p_all = np.zeros((H, T))
    for h in range(H):
        g = h // group
        s = (K[g] @ q[h]) / np.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        p_all[h] = p
        out[h] = p @ V[g]
    return out, p_all


def step_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, k_cache_bits: np.ndarray, v_cache_bits: np.ndarray,
                   pos: int, theta: float = 10000.0) -> Tuple[np.ndarray, np.ndarray]:
    """One layer's attention in a decode step at position pos.

    q [H*d], k and v [H_kv*d]: the projection outputs, rounded to bf16 as the
    cache stores them; q and k turned by rope_bf16 at pos; k and v written into
    copies of the caches (bf16 [H_kv, >= pos + 1, d]) at pos; then
    attention_decode over positions 0 .. pos. Returns (out [H*d] fp64, the
    updated (k, v) cache rows at pos as bf16 [H_kv, d] each, stacked).
    """
    Hkv, _, d = k_cache_bits.shape
    H = q.size // d
    qb = rope_bf16(f64_to_bf16_bits(np.asarray(q, np.float64)).reshape(H, d), pos, theta)
    kb = rope_bf16(f64_to_bf16_bits(np.asarray(k, np.float64)).reshape(Hkv, d), pos, theta)
    vb = f64_to_bf16_bits(np.asarray(v, np.float64)).reshape(Hkv, d)
    kc = k_cache_bits.copy()
    vc = v_cache_bits.copy()
    kc[:, pos, :] = kb
    vc[:, pos, :] = vb
    out, _ = attention_decode(qb, kc, vc, pos + 1)
    return out.reshape(-1), np.stack([kb, vb])

