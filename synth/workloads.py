"""Seeded input generators for VBQ matrices and activations.

Every array here is drawn from numpy's PCG64 with a SeedSequence keyed by
(seed, stream...), so a workload is fully fixed by its seed and its name.

Distributions (the synthetic stand-in for trained allocations; the VBQ abstract
on the "Variable Bit-width Quantization" page reports 69% of groups at 1 bit, an
LM head near 1.09 bits and a first MLP block near 2.5 bits):

* per-group bit-width b in {1,2,4,8}: iid categorical with the given
  probabilities, drawn by inverse CDF on a uniform double;
* codes q: uniform on [0, 2^b - 1] (a uniform byte masked to its low b bits);
* scales: uniform on [0.01, 0.05] in double, rounded to fp16 (round to nearest
  even, numpy's double -> half conversion);
* activations x: N(0, 1) drawn in double, cast to fp32, rounded to bf16 (round
  to nearest even).

The layout of the outputs is the logical one that the packer consumes:
codes uint8 [N, K] row-major, bits uint8 [N, K/64], scales uint16 [N, K/64]
holding fp16 bit patterns.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

GROUP = 64
PROJS = ("q", "k", "v", "o", "gate", "up", "down")
HEAD = "head"

# Bit-width probabilities {bits: P}.
CONFIG0_PROBS: Dict[int, float] = {1: 0.69, 2: 0.15, 4: 0.11, 8: 0.05}
LAYER0_MLP_PROBS: Dict[int, float] = {1: 0.35, 2: 0.25, 4: 0.25, 8: 0.15}
HEAD_PROBS: Dict[int, float] = {1: 0.97, 2: 0.02, 4: 0.01, 8: 0.0}

_STREAM_MATRIX = 0
_STREAM_MODEL = 1
_STREAM_X = 2
_STREAM_STRESS = 3


@dataclass(frozen=True)
class VbqMatrixInputs:
    """Logical (unpacked) VBQ matrix: codes, per-group bit-widths and scales."""

    codes: np.ndarray   # uint8 [N, K], code q of each weight
    bits: np.ndarray    # uint8 [N, K/64], bit-width of each group
    scales: np.ndarray  # uint16 [N, K/64], fp16 bit pattern of each group scale

    @property
    def N(self) -> int:
        return int(self.codes.shape[0])

    @property
    def K(self) -> int:
        return int(self.codes.shape[1])


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, stream)])))


def draw_bits(rng: np.random.Generator, n: int, g: int, probs: Dict[int, float]) -> np.ndarray:
    """Categorical bit-widths by inverse CDF on uniform doubles."""
    u = rng.random((n, g))
    out = np.full((n, g), 8, dtype=np.uint8)
    cum = 0.0
    # Assign from the widest class down so that narrower classes overwrite.
    edges = []
    for b in (1, 2, 4):
        cum += float(probs.get(b, 0.0))
        edges.append((b, cum))
    for b, edge in reversed(edges):
        out[u < edge] = b
    return out


def draw_codes(rng: np.random.Generator, bits: np.ndarray) -> np.ndarray:
    """Uniform codes in [0, 2^b - 1] for each group's bit-width b."""
    n, g = bits.shape
    total = n * g * GROUP
    raw = rng.bit_generator.random_raw((total + 7) // 8).view(np.uint8)[:total]
    mask = ((np.uint16(1) << bits.astype(np.uint16)) - np.uint16(1)).astype(np.uint8)
    codes = raw.reshape(n, g, GROUP) & mask[:, :, None]
    return codes.reshape(n, g * GROUP)


def draw_scales(rng: np.random.Generator, n: int, g: int, lo: float = 0.01, hi: float = 0.05) -> np.ndarray:
    return rng.uniform(lo, hi, size=(n, g)).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Used only to produce inputs; finite values only.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gen_matrix(n: int, k: int, probs: Dict[int, float], seed: int = 0,
               stream: Sequence[int] = (_STREAM_MATRIX, 0)) -> VbqMatrixInputs:
    """One VBQ matrix [n, k] with iid per-group bit-widths drawn from ``probs``."""
    if k % GROUP:
        raise ValueError("K must be a multiple of 64")
    g = k // GROUP
    rng = _rng(seed, *stream)
    bits = draw_bits(rng, n, g, probs)
    codes = draw_codes(rng, bits)
    scales = draw_scales(rng, n, g)
    return VbqMatrixInputs(codes=codes, bits=bits, scales=scales)


def gen_matrix_with_bits(bits: np.ndarray, seed: int, stream: Sequence[int]) -> VbqMatrixInputs:
    rng = _rng(seed, *stream)
    n, g = bits.shape
    codes = draw_codes(rng, bits)
    scales = draw_scales(rng, n, g)
    return VbqMatrixInputs(codes=codes, bits=np.ascontiguousarray(bits, dtype=np.uint8), scales=scales)


STRESS_CASES = ("a", "b", "c", "d", "e")


def stress_bits(case: str, n: int, k: int, seed: int = 0) -> np.ndarray:
    """Bit maps of the allocation-stress cases on an n x k matrix.

    a: all 1-bit; b: all 8-bit; c: iid with CONFIG0_PROBS;
    d: rows [0, n/2) draw P(4)=P(8)=0.5 (mean 6 bits), rows [n/2, n) are 1-bit;
    e: the first quarter of the groups of every row are 8-bit, the rest 1-bit.
    """
    g = k // GROUP
    rng = _rng(seed, _STREAM_STRESS, ord(case))
    if case == "a":
        return np.full((n, g), 1, np.uint8)
    if case == "b":
        return np.full((n, g), 8, np.uint8)
    if case == "c":
        return draw_bits(rng, n, g, CONFIG0_PROBS)
    if case == "d":
        bits = np.full((n, g), 1, np.uint8)
        half = n // 2
        bits[:half] = draw_bits(rng, half, g, {1: 0.0, 2: 0.0, 4: 0.5, 8: 0.5})
        return bits
    if case == "e":
        bits = np.full((n, g), 1, np.uint8)
        bits[:, : g // 4] = 8
        return bits
    raise ValueError(f"unknown stress case {case!r}")


def gen_stress(case: str, n: int = 8192, k: int = 8192, seed: int = 0) -> VbqMatrixInputs:
    bits = stress_bits(case, n, k, seed)
    return gen_matrix_with_bits(bits, seed, (_STREAM_STRESS, ord(case), 1))


def gen_x(k: int, seed: int = 0, batch: Optional[int] = None, tag: int = 0) -> np.ndarray:
    """bf16 activations ~N(0,1) as uint16 bit patterns; shape [k] or [batch, k]."""
    rng = _rng(seed, _STREAM_X, tag)
    shape = (k,) if batch is None else (batch, k)
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


@dataclass(frozen=True)
class ModelShape:
    """Shapes of a decoder-only stack whose projections are VBQ matrices."""

    name: str
    n_layers: int
    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    layer0_mlp_probs: Optional[Dict[int, float]]
    head_probs: Dict[int, float]
    body_probs: Dict[int, float] = None  # type: ignore[assignment]

    def probs(self) -> Dict[int, float]:
        return self.body_probs if self.body_probs is not None else CONFIG0_PROBS


def model_1b() -> ModelShape:
    """1.0B-shaped stack: 16 layers, d=2048, MHA 16x128, SwiGLU 5632, vocab 32000."""
    return ModelShape("vbq-1b", 16, 2048, 16, 16, 128, 5632, 32000, LAYER0_MLP_PROBS, HEAD_PROBS)


def model_9b() -> ModelShape:
    """9B-shaped stack: 32 layers, d=4096, GQA 32q/8kv x128, SwiGLU 14336, vocab 128256."""
    return ModelShape("vbq-9b", 32, 4096, 32, 8, 128, 14336, 128256, None, HEAD_PROBS)


def model_tiny() -> ModelShape:
    """A small stack with the same structure (GQA, SwiGLU), for fast parity runs."""
    return ModelShape("vbq-tiny", 2, 256, 4, 2, 64, 384, 1000, LAYER0_MLP_PROBS, HEAD_PROBS)


def model_matrix_shape(m: ModelShape, proj: str) -> Tuple[int, int]:
    """(N, K) = (out, in) of one projection."""
    hq = m.n_heads * m.head_dim
    hkv = m.n_kv_heads * m.head_dim
    return {
        "q": (hq, m.d), "k": (hkv, m.d), "v": (hkv, m.d), "o": (m.d, hq),
        "gate": (m.d_ff, m.d), "up": (m.d_ff, m.d), "down": (m.d, m.d_ff),
        HEAD: (m.vocab, m.d),
    }[proj]


def model_matrix_probs(m: ModelShape, layer: int, proj: str) -> Dict[int, float]:
    if proj == HEAD:
        return m.head_probs
    if layer == 0 and proj in ("gate", "up", "down") and m.layer0_mlp_probs is not None:
        return m.layer0_mlp_probs
    return m.probs()


def gen_model_matrix(m: ModelShape, layer: int, proj: str, seed: int = 0) -> VbqMatrixInputs:
    """One projection of a model; the head is (layer = n_layers, proj = 'head')."""
    n, k = model_matrix_shape(m, proj)
    pid = 7 if proj == HEAD else PROJS.index(proj)
    return gen_matrix(n, k, model_matrix_probs(m, layer, proj), seed, (_STREAM_MODEL, layer, pid))


def model_matrix_list(m: ModelShape):
    """[(layer, proj)] in the order the decode step consumes them, head last."""
    out = [(l, p) for l in range(m.n_layers) for p in PROJS]
    out.append((m.n_layers, HEAD))
    return out
