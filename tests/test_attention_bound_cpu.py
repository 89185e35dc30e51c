"""The attention parity bound on the CPU: an fp32 emulation of the split-KV arithmetic stays inside it
against the fp64 oracle, on the GPU tests' shapes and span counts and on sharp scores, and planted
mistakes in the emulation break it (CPU only)."""

import numpy as np
import pytest

from oracle import attention_oracle as A
from oracle.vbq_oracle import f64_to_bf16_bits
from tests import parity_bound as PB


def _case(H, Hkv, d, T, seed, qscale=1.0):
    rng = np.random.default_rng(seed)
    q = f64_to_bf16_bits(rng.standard_normal((H, d)) * qscale)
    k = f64_to_bf16_bits(rng.standard_normal((Hkv, T, d)))
    v = f64_to_bf16_bits(rng.standard_normal((Hkv, T, d)))
    return q, k, v


def _ratio(q, k, v, T, emu):
    ref, p = A.attention_decode(q, k, v, T)
    return np.abs(emu - ref) / PB.attention_bound(q, k, v, T, p)


@pytest.mark.parametrize("H,Hkv,d,T,nparts", [(32, 8, 128, 1, 55), (32, 8, 128, 200, 55), (32, 8, 128, 4096, 55),
                                              (16, 16, 64, 300, 27), (12, 4, 64, 129, 64), (8, 1, 128, 65, 64),
                                              (8, 2, 128, 3000, 1), (8, 2, 128, 3000, 7)])
@pytest.mark.parametrize("qscale", [1.0, 8.0])
def test_emulated_attention_within_bound(H, Hkv, d, T, nparts, qscale):
    q, k, v = _case(H, Hkv, d, T, seed=H + T + d, qscale=qscale)
    r = _ratio(q, k, v, T, PB.emulate_attention(q, k, v, T, nparts))
    assert r.max() <= 1.0, float(r.max())


@pytest.mark.parametrize("mistake", ["drop_last", "scale_by_d"])
def test_planted_mistakes_break_the_bound(mistake):
    H, Hkv, d, T = 8, 2, 64, 129
    q, k, v = _case(H, Hkv, d, T, seed=5)
    r = _ratio(q, k, v, T, PB.emulate_attention(q, k, v, T, 3, **{mistake: True}))
    assert r.max() > 1.0


def test_bound_is_far_below_the_values():
    """The bound is a small fraction of sum_j p_j |v_j| (it can catch a wrong weight or position)."""
    H, Hkv, d, T = 8, 2, 128, 4096
    q, k, v = _case(H, Hkv, d, T, seed=6)
    _, p = A.attention_decode(q, k, v, T)
    from oracle.vbq_oracle import bf16_bits_to_f64
    scale = np.stack([p[h] @ np.abs(bf16_bits_to_f64(v)[h // 4, :T]) for h in range(H)])
    assert (PB.attention_bound(q, k, v, T, p) / scale).max() < 2e-3
