"""Pins of the attention oracle (CPU): closed forms, special cases and invariants.

Each check takes the oracle's three functions as M, so that
test_planted_mistakes_fail_a_pin can run the same checks on copies of the
oracle with one step done the wrong way."""

import types

import numpy as np
import pytest

from oracle import attention_oracle as A
from oracle.vbq_oracle import bf16_bits_to_f64, f64_to_bf16_bits


def _bf16(rng, shape, scale=1.0):
    return f64_to_bf16_bits(rng.standard_normal(shape) * scale)


def check_rope_at_position_zero_is_the_identity(M=A):
    x = _bf16(np.random.default_rng(1), (5, 128))
    assert np.array_equal(M.rope_bf16(x, 0), x)


def check_rope_hand_case(M=A):
    # d = 2: the single pair turns by pos radians; d = 4, theta = 100: pair 1 turns by pos / 10.
    y = M.rope_f64(np.array([[1.0, 0.0]]), 1)
    assert np.allclose(y, [[np.cos(1.0), np.sin(1.0)]], rtol=0, atol=1e-15)
    y = M.rope_f64(np.array([[0.0, 2.0, 0.0, 0.0]]), 3, theta=100.0)
    assert np.allclose(y, [[0.0, 2.0 * np.cos(0.3), 0.0, 2.0 * np.sin(0.3)]], rtol=0, atol=1e-15)


def check_rope_keeps_each_pair_norm_and_composes(M=A):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 64))
    y = M.rope_f64(x, 777)
    half = 32
    assert np.allclose(np.hypot(y[:, :half], y[:, half:]), np.hypot(x[:, :half], x[:, half:]), rtol=1e-13)
    assert np.allclose(M.rope_f64(M.rope_f64(x, 100), 23), M.rope_f64(x, 123), rtol=0, atol=1e-11)


def check_rope_bf16_is_the_fp64_rotation_rounded(M=A):
    rng = np.random.default_rng(3)
    x = _bf16(rng, (3, 128))
    y = M.rope_bf16(x, 4095)
    ref = M.rope_f64(bf16_bits_to_f64(x), 4095)
    err = np.abs(bf16_bits_to_f64(y) - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-38)


def check_attention_over_one_position_returns_its_value(M=A):
    rng = np.random.default_rng(4)
    q, k, v = _bf16(rng, (8, 64)), _bf16(rng, (2, 5, 64)), _bf16(rng, (2, 5, 64))
    out, p = M.attention_decode(q, k, v, 1)
    V = bf16_bits_to_f64(v)
    assert np.array_equal(p, np.ones((8, 1)))
    assert np.array_equal(out, np.repeat(V[:, 0, :], 4, axis=0))


def check_zero_query_averages_the_values(M=A):
    rng = np.random.default_rng(5)
    q = np.zeros((4, 128), np.uint16)
    k, v = _bf16(rng, (4, 37, 128)), _bf16(rng, (4, 37, 128))
    out, _ = M.attention_decode(q, k, v, 30)
    assert np.allclose(out, bf16_bits_to_f64(v)[:, :30, :].mean(axis=1), rtol=0, atol=1e-14)


def check_dominant_score_picks_its_value(M=A):
    rng = np.random.default_rng(6)
    d, T, j = 64, 50, 17
    q = np.zeros((2, d), np.uint16)
    q[:, 0] = f64_to_bf16_bits(np.array([1.0, 1.0]))
    k = np.zeros((1, T, d), np.uint16)
    k[0, j, 0] = f64_to_bf16_bits(np.array([65536.0]))[0]  # score 8192 against 0: exp(8192) overflows fp64
    v = _bf16(rng, (1, T, d))
    out, p = M.attention_decode(q, k, v, T)
    assert p[0, j] == 1.0
    assert np.allclose(out, bf16_bits_to_f64(v)[0, j][None, :], rtol=0, atol=1e-200)


def check_two_positions_closed_form(M=A):
    # q = e_0, k_0 = 8 e_0, k_1 = 0, d = 64: scores 8 / sqrt(64) = 1 and 0, so p_0 = 1 / (1 + e^-1).
    d = 64
    q = np.zeros((1, d), np.uint16)
    q[0, 0] = f64_to_bf16_bits(np.array([1.0]))[0]
    k = np.zeros((1, 2, d), np.uint16)
    k[0, 0, 0] = f64_to_bf16_bits(np.array([8.0]))[0]
    v = np.zeros((1, 2, d), np.uint16)
    v[0, 0, :] = f64_to_bf16_bits(np.full(d, 3.0))
    v[0, 1, :] = f64_to_bf16_bits(np.full(d, -1.0))
    out, p = M.attention_decode(q, k, v, 2)
    p0 = 1.0 / (1.0 + np.exp(-1.0))
    assert abs(p[0, 0] - p0) < 1e-15
    assert np.allclose(out[0], 3.0 * p0 - (1.0 - p0), rtol=0, atol=1e-14)


def check_query_heads_read_their_own_kv_head(M=A):
    rng = np.random.default_rng(7)
    H, Hkv, d, T = 8, 2, 64, 9
    q = _bf16(rng, (H, d))
    q[1] = q[0]                                   # heads 0 and 1 share kv head 0
    k, v = _bf16(rng, (Hkv, T, d)), _bf16(rng, (Hkv, T, d))
    out, _ = M.attention_decode(q, k, v, T)
    assert np.array_equal(out[0], out[1])
    v2 = v.copy()
    v2[1] = _bf16(rng, (T, d))                     # change kv head 1 only
    out2, _ = M.attention_decode(q, k, v2, T)
    assert np.array_equal(out[:4], out2[:4]) and not np.allclose(out[4:], out2[4:])


def check_positions_are_a_set(M=A):
    rng = np.random.default_rng(8)
    q, k, v = _bf16(rng, (4, 128)), _bf16(rng, (1, 40, 128)), _bf16(rng, (1, 40, 128))
    perm = rng.permutation(40)
    a, _ = M.attention_decode(q, k, v, 40)
    b, _ = M.attention_decode(q, k[:, perm], v[:, perm], 40)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)


CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__[6:])
def test_pin(check):
    check(A)


# ---- planted mistakes ----

def _rope_variant(kind):
    def rope_f64(x, pos, theta=10000.0):
        x = np.asarray(x, dtype=np.float64)
        d = x.shape[-1]
        half = d // 2
        i = np.arange(half, dtype=np.float64)
        expo = -1.0 * i / d if kind == "exponent_-i/d" else -2.0 * i / d
        ang = float(pos) * np.power(float(theta), expo)
        if kind == "angle_sign":
            ang = -ang
        c, s = np.cos(ang), np.sin(ang)
        if kind == "interleaved_pairs":
            x0, x1 = x[..., 0::2], x[..., 1::2]
            y = np.empty_like(x)
            y[..., 0::2], y[..., 1::2] = x0 * c - x1 * s, x0 * s + x1 * c
            return y
        x0, x1 = x[..., :half], x[..., half:]
        return np.concatenate([x0 * c - x1 * s, x0 * s + x1 * c], axis=-1)
    return rope_f64


def _attention_variant(kind):
    def attention_decode(q_bits, k_bits, v_bits, T):
        q = bf16_bits_to_f64(q_bits)
        K = bf16_bits_to_f64(k_bits)[:, :T, :]
        V = bf16_bits_to_f64(v_bits)[:, :T, :]
        H, d = q.shape
        Hkv = K.shape[0]
        group = H // Hkv
        out, p_all = np.zeros((H, d)), np.zeros((H, T))
        for h in range(H):
            g = h % Hkv if kind == "head_modulo" else h // group
            s = K[g] @ q[h] if kind == "no_scale" else (K[g] @ q[h]) / np.sqrt(d)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.exp(s) if kind == "no_max_shift" else np.exp(s - s.max())
                p = p / p.sum()
            if kind == "values_last_T":
                out[h] = p @ bf16_bits_to_f64(v_bits)[g, -T:, :]
            else:
                out[h] = p @ V[g]
            p_all[h] = p
        return out, p_all
    return attention_decode


def _oracle_with(rope=None, attention=None):
    rope_f64 = rope or A.rope_f64

    def rope_bf16(x_bits, pos, theta=10000.0):
        y = rope_f64(bf16_bits_to_f64(x_bits), pos, theta)
        return f64_to_bf16_bits(y.astype(np.float32).astype(np.float64))
    return types.SimpleNamespace(rope_f64=rope_f64, rope_bf16=rope_bf16,
                                 attention_decode=attention or A.attention_decode)


MUTANTS = {
    "rope_exponent_-i/d": lambda: _oracle_with(rope=_rope_variant("exponent_-i/d")),
    "rope_angle_sign": lambda: _oracle_with(rope=_rope_variant("angle_sign")),
    "rope_interleaved_pairs": lambda: _oracle_with(rope=_rope_variant("interleaved_pairs")),
    "attention_head_modulo": lambda: _oracle_with(attention=_attention_variant("head_modulo")),
    "attention_no_scale": lambda: _oracle_with(attention=_attention_variant("no_scale")),
    "attention_no_max_shift": lambda: _oracle_with(attention=_attention_variant("no_max_shift")),
    "attention_values_last_T": lambda: _oracle_with(attention=_attention_variant("values_last_T")),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(name):
    M = MUTANTS[name]()
    failed = []
    for check in CHECKS:
        try:
            check(M)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the mutant {name}"


def test_step_attention_at_position_zero_is_the_position_zero_rule():
    """At pos 0 the rotation is the identity and the softmax is over one key: each query head returns
    its kv head's v, rounded to bf16, whatever the cache held."""
    from oracle import vbq_oracle as O
    rng = np.random.default_rng(9)
    H, Hkv, d = 8, 2, 64
    q, k, v = rng.standard_normal(H * d), rng.standard_normal(Hkv * d), rng.standard_normal(Hkv * d)
    kc, vc = _bf16(rng, (Hkv, 5, d)), _bf16(rng, (Hkv, 5, d))
    out, rows = A.step_attention(q, k, v, kc, vc, 0)
    vb = bf16_bits_to_f64(f64_to_bf16_bits(v))
    assert np.array_equal(out, O.attention_pos0(vb, H, Hkv, d))
    assert np.array_equal(rows[0], f64_to_bf16_bits(k).reshape(Hkv, d))
