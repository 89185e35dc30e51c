"""Plant plausible mistakes in copies of the oracle (CPU) and check the pins catch each.

Each mutant rewrites one step of the oracle's dequantize or dot product the
wrong way. Every mutant must fail at least one check in tests/oracle_pins.py.
"""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import bf16_bits_to_f32
from tests import oracle_pins as P

GROUP = 64


def _mut_dequant(kind):
    def dq(codes, bits, scales):
        n, k = codes.shape
        g = k // GROUP
        s = scales.view(np.float16).astype(np.float32)
        b = bits.astype(np.int64)
        c = ((1 << b) - 1) / 2.0
        if kind == "offset_2^b/2":
            c = (1 << b) / 2.0
        if kind == "offset_2^(b-1)-1":
            c = (1 << (b - 1)) - 1.0
        q = codes.reshape(n, g, GROUP).astype(np.float32)
        if kind == "scale_dropped":
            s = np.ones_like(s)
        if kind == "scale_transposed":
            # group index taken as k % G instead of k // 64
            kk = np.arange(k)
            w = s[:, kk % g] * (codes.astype(np.float32) - c.astype(np.float32)[:, kk % g])
            return w.astype(np.float32)
        if kind == "sign_flipped":
            w = s[:, :, None] * (c.astype(np.float32)[:, :, None] - q)
        else:
            w = s[:, :, None] * (q - c.astype(np.float32)[:, :, None])
        if kind == "bf16_weights":
            w = O.bf16_round(w).astype(np.float32)
        return w.reshape(n, k).astype(np.float32)
    return dq


def _gemv_from(dq, acc=np.float64, x_fix=None):
    def gv(codes, bits, scales, x_bits):
        W = dq(codes, bits, scales).astype(acc)
        x = bf16_bits_to_f32(x_bits).astype(acc)
        if x_fix is not None:
            x = x_fix(x)
        return (W @ x).astype(np.float64)
    return gv


MUTANTS = {
    "offset_2^b/2": lambda: (_mut_dequant("offset_2^b/2"), None),
    "offset_2^(b-1)-1": lambda: (_mut_dequant("offset_2^(b-1)-1"), None),
    "scale_dropped": lambda: (_mut_dequant("scale_dropped"), None),
    "scale_transposed": lambda: (_mut_dequant("scale_transposed"), None),
    "sign_flipped": lambda: (_mut_dequant("sign_flipped"), None),
    "bf16_weights": lambda: (_mut_dequant("bf16_weights"), None),
    "fp32_accumulation": lambda: (O.dequant, _gemv_from(O.dequant, acc=np.float32)),
    "x_reversed": lambda: (O.dequant, _gemv_from(O.dequant, x_fix=lambda x: x[::-1].copy())),
    "x_last_dropped": lambda: (O.dequant, _gemv_from(O.dequant, x_fix=lambda x: np.concatenate([x[:-1], [0.0]]))),
}


def _caught(dq, gv):
    checks = [
        lambda: P.check_dequant_bruteforce(dq),
        lambda: P.check_gemv_bruteforce(gv),
        lambda: P.check_closed_form_1bit(gv),
        lambda: P.check_closed_form_8bit(gv),
        lambda: P.check_onehot_identity(gv),
        lambda: P.check_linearity(gv),
    ]
    failures = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failures += 1
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    dq, gv = MUTANTS[name]()
    if gv is None:
        gv = _gemv_from(dq)
    assert _caught(dq, gv) >= 1, name


def test_real_oracle_passes_all():
    assert _caught(O.dequant, O.gemv) == 0


# ---- row norms: the denominator of every parity bar ----

def _norms_from(kind):
    def rn(codes, bits, scales):
        W = O.dequant(codes, bits, scales).astype(np.float64)
        if kind == "squared_norm":
            return (W * W).sum(axis=1)
        if kind == "l1_norm":
            return np.abs(W).sum(axis=1)
        if kind == "mean_square_root":
            return np.sqrt((W * W).mean(axis=1))
        raise ValueError(kind)
    return rn


def _norms_caught(rn):
    failures = 0
    for c in (lambda: P.check_row_norms_bruteforce(rn), lambda: P.check_row_norms_hand(rn)):
        try:
            c()
        except AssertionError:
            failures += 1
    return failures


@pytest.mark.parametrize("kind", ["squared_norm", "l1_norm", "mean_square_root"])
def test_row_norm_mutant_is_caught(kind):
    assert _norms_caught(_norms_from(kind)) >= 1, kind


def test_real_row_norms_pass():
    assert _norms_caught(O.row_norms) == 0
