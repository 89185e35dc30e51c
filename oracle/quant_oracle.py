"""CPU oracle for the divergence measurement: dense weights onto the VBQ grid, and the distance
between two models' next-token distributions. Plain numpy, fp64.

TEST INFRASTRUCTURE ONLY. Only the tests and bench.py may import this module. The library never
calls it, and it shares no code with the CUDA path or the library's host code.

The VBQ abstract ("Variable Bit-width Quantization: Learning Per-Group Precision for
'Bigger-but-Smaller' Language Models") analyses how a quantized model's output distribution moves
from the dense one with the KL divergence and the argmax-flip rate. The pages learn the weights and
the allocation; given an allocation, the plainest encoding of dense weights onto the grid
w = s (q - c_b), c_b = (2^b - 1)/2, is absmax round-to-nearest per group of 64, which this module
writes out:

* s = max|w| / c_b, rounded to fp16 (nearest, ties to even);
* q = the nearest integer (ties to even) to w / s + c_b, clipped to [0, 2^b - 1]; q = 0 where s = 0.

KL(P || Q) = sum_i P_i (log P_i - log Q_i) for P = softmax(dense logits), Q = softmax(test
logits); a flip is argmax P != argmax Q.

Parity pins: tests/test_quant_oracle.py (grid round trip, the error bound, zero and 1-bit groups,
brute-force nearest codes on the stored grid, the nearest fp16 scale, KL and log-softmax closed
forms, the flip rule), each checked to catch planted mistakes in a copy of this module.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

GROUP = 64


def quantize_rtn(W: np.ndarray, bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Dense [N, K] weights at the bit map [N, K/64] -> (codes uint8 [N, K], fp16 scale bits [N, K/64])."""
    W = np.asarray(W, dtype=np.float32).astype(np.float64)
    n, k = W.shape
    g = k // GROUP
    Wg = W.reshape(n, g, GROUP)
    b = np.asarray(bits, dtype=np.int64)
    c = (np.ldexp(1.0, b) - 1.0) / 2.0
    qmax = np.ldexp(1.0, b) - 1.0
    s16 = (np.abs(Wg).max(axis=2) / c).astype(np.float16)
    s = s16.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, :, None] > 0, np.rint(Wg / s[:, :, None] + c[:, :, None]), 0.0)
    q = np.clip(q, 0.0, qmax[:, :, None])
    return q.reshape(n, k).astype(np.uint8), s16.view(np.uint16)


def log_softmax(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    return z - m - np.log(np.exp(z - m).sum(axis=-1, keepdims=True))


def kl_and_flips(dense_logits: np.ndarray, test_logits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per input row: KL(softmax(dense) || softmax(test)) and whether the argmax differs."""
    lp = log_softmax(dense_logits)
    lq = log_softmax(test_logits)
    kl = (np.exp(lp) * (lp - lq)).sum(axis=-1)
    flips = np.argmax(dense_logits, axis=-1) != np.argmax(test_logits, axis=-1)
    return kl, flips
