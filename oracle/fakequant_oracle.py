"""CPU oracle for the training-side fake quantization (Gumbel-Softmax mixture over {1,2,4,8} bits
per group of 64, straight-through backward). Plain numpy.

TEST INFRASTRUCTURE ONLY. Only the tests may import this module; the library never calls it, and it
shares no code with the CUDA path.

The VBQ abstract ("Variable Bit-width Quantization: Learning Per-Group Precision for
'Bigger-but-Smaller' Language Models") learns each group's precision with a Gumbel-Softmax
relaxation over precision logits, optimised alternately with the weights, and passes gradients
through the rounding with the straight-through estimator. The pages give no formulas; this module
writes out the plainest reading, with the level decisions in fp32 (the precision the kernel takes
them in) and everything else in fp64:

* Q_b(w) = s_b (q - c_b), c_b = (2^b - 1)/2, s_b = max|w_g| / c_b, q = rint(w r_b + c_b) with
  r_b = c_b / max|w_g|, clipped to [0, 2^b - 1] (each fp32 operation rounded once); Q_b = 0 for an
  all-zero group;
* pi_b = softmax_b((alpha_gb - log(-log u_gb)) / tau); W_mix = sum_b pi_b Q_b(W);
* backward for G = dL/dW_mix: dW = G; dalpha_b = (pi_b / tau) (D_b - sum_b' pi_b' D_b'),
  D_b = sum over the group of G Q_b(W).

Parity pins: tests/test_fakequant_oracle.py (one-hot mixtures, on-grid weights, the Gumbel
transform's closed form, softmax(alpha / tau) under equal noise, a two-width split, the closed-form
gradient against finite differences of the forward, the straight-through identity), each checked to
catch planted mistakes in a copy of this module.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

GROUP = 64
BITS = (1, 2, 4, 8)


def levels(W: np.ndarray) -> np.ndarray:
    """Q_b(W) for the four bit-widths: [4, N, K], fp32 values (the kernel's arithmetic)."""
    W = np.asarray(W, dtype=np.float32)
    n, k = W.shape
    Wg = W.reshape(n, k // GROUP, GROUP)
    mx = np.abs(Wg).max(axis=2, keepdims=True)
    out = np.zeros((4, n, k // GROUP, GROUP), np.float32)
    for i, b in enumerate(BITS):
        qmax = np.float32((1 << b) - 1)
        c = np.float32(0.5) * qmax
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            s = mx / c
            r = c / mx
            q = np.clip(np.rint(Wg * r + c), np.float32(0), qmax)
            v = s * (q - c)
        out[i] = np.where(mx > 0, v, np.float32(0))
    return out.reshape(4, n, k)


def mixture(alpha: np.ndarray, u: np.ndarray, tau: float) -> np.ndarray:
    """pi [N, G, 4] in fp64."""
    z = (np.asarray(alpha, np.float64) - np.log(-np.log(np.asarray(u, np.float64)))) / tau
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def forward(W, alpha, u, tau) -> np.ndarray:
    Q = levels(W).astype(np.float64)               # [4, N, K]
    pi = mixture(alpha, u, tau)                    # [N, G, 4]
    piw = np.repeat(np.moveaxis(pi, -1, 0), GROUP, axis=2)  # [4, N, K]
    return (piw * Q).sum(axis=0)


def backward(W, alpha, u, tau, G) -> Tuple[np.ndarray, np.ndarray]:
    Q = levels(W).astype(np.float64)
    pi = mixture(alpha, u, tau)
    n, k = np.asarray(W).shape
    Gd = np.asarray(G, np.float64)
    D = (Gd[None] * Q).reshape(4, n, k // GROUP, GROUP).sum(axis=3)  # [4, N, G]
    D = np.moveaxis(D, 0, -1)                                        # [N, G, 4]
    mean = (pi * D).sum(axis=-1, keepdims=True)
    return Gd.copy(), pi / tau * (D - mean)
