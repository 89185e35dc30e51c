"""The oracle against what the mathematics fixes (CPU only)."""

import json
import os

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import (CONFIG0_PROBS, bf16_bits_to_f32, f32_to_bf16_bits, gen_matrix, gen_stress,
                   gen_x, stress_bits)
from tests import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dequant_bruteforce_exact(seed):
    P.check_dequant_bruteforce(O.dequant, seed)


@pytest.mark.parametrize("seed", [0, 1])
def test_gemv_bruteforce_exact(seed):
    P.check_gemv_bruteforce(O.gemv, seed)


def test_closed_form_1bit():
    P.check_closed_form_1bit(O.gemv)


def test_closed_form_8bit():
    P.check_closed_form_8bit(O.gemv)


def test_onehot_identity():
    P.check_onehot_identity(O.gemv)


def test_linearity():
    P.check_linearity(O.gemv)


def test_storage_invariants():
    P.check_storage(O.storage_bytes)


@pytest.mark.parametrize("seed", [0, 1])
def test_row_norms_bruteforce_exact(seed):
    P.check_row_norms_bruteforce(O.row_norms, seed)


def test_row_norms_hand_matrix():
    P.check_row_norms_hand(O.row_norms)


def test_row_chunks_cover_rows_in_order():
    # rows per chunk = budget // (8 K), at least 1; the chunks tile [0, n) in order
    for n, k, budget in [(10, 64, 8 * 64 * 3), (7, 128, 1), (5, 64, 1 << 30), (0, 64, 100)]:
        chunks = list(O._row_chunks(n, k, budget))
        rows = max(1, budget // (8 * k))
        assert [r0 for r0, _ in chunks] == list(range(0, n, rows))
        assert all(r1 - r0 == min(rows, n - r0) for r0, r1 in chunks)


def test_gemm_and_row_norms_over_several_chunks(monkeypatch):
    # The same rows through at least three chunks give the same values: rows are independent.
    m = gen_matrix(37, 256, CONFIG0_PROBS, seed=8)
    X = gen_x(256, seed=8, batch=2)
    Y1, n1 = O.gemm(m.codes, m.bits, m.scales, X), O.row_norms(m.codes, m.bits, m.scales)
    real = O._row_chunks
    seen = []

    def small(n, k, budget_bytes=0):
        out = list(real(n, k, 8 * k * 10))   # 10 rows per chunk
        seen.append(len(out))
        return iter(out)

    monkeypatch.setattr(O, "_row_chunks", small)
    Y2, n2 = O.gemm(m.codes, m.bits, m.scales, X), O.row_norms(m.codes, m.bits, m.scales)
    assert min(seen) >= 3
    np.testing.assert_allclose(Y2, Y1, rtol=1e-15, atol=0.0)
    assert np.array_equal(n2, n1)


def test_gemm_columns_are_gemvs():
    m = gen_matrix(40, 256, CONFIG0_PROBS, seed=7)
    X = gen_x(256, seed=7, batch=3)
    Y = O.gemm(m.codes, m.bits, m.scales, X)
    for j in range(3):
        assert np.array_equal(Y[j], O.gemv(m.codes, m.bits, m.scales, X[j]))


def test_dequant_rejects_bad_inputs():
    m = gen_matrix(4, 128, CONFIG0_PROBS, seed=1)
    bad_bits = m.bits.copy()
    bad_bits[0, 0] = 3
    with pytest.raises(ValueError):
        O.dequant(m.codes, bad_bits, m.scales)
    bad_codes = m.codes.copy()
    one = np.argwhere(m.bits == 1)[0]
    bad_codes[one[0], one[1] * 64] = 2
    with pytest.raises(ValueError):
        O.dequant(bad_codes, m.bits, m.scales)
    with pytest.raises(ValueError):
        O.dequant(m.codes[:, :100], m.bits, m.scales)


def test_normalized_error_definition():
    w = np.array([3.0, 4.0])
    x = f32_to_bf16_bits(np.array([1.0, 0.0, 0.0], np.float32))  # ||x|| = 1
    e = O.normalized_error(np.array([1.0, 2.5]), np.array([0.0, 2.0]), w, x)
    assert e == pytest.approx(max(1.0 / 3.0, 0.5 / 4.0))


# ---- bf16 rounding: against torch's own float64 -> bfloat16 conversion ----

def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        # exact ties between neighbouring bf16 values, both parities
        (1.0 + (2 * np.arange(1, 200) + 1) * 2.0 ** -8) * 2.0 ** -7,
        -(1.0 + (2 * np.arange(1, 200)) * 2.0 ** -8 + 2.0 ** -8),
        np.array([0.0, -0.0, 1.0, 2.0 ** -126, 3.0 * 2.0 ** -130, 1e-40]),
    ])
    ours = O.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    bits = O.f64_to_bf16_bits(v[:1000])
    assert np.array_equal(bf16_bits_to_f32(bits).astype(np.float64), ref[:1000])


def test_fp16_scale_decode_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    ours = O.f16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


# ---- generator statistics (the allocation the synthetic workloads stand in for) ----

def test_generator_class_frequencies():
    m = gen_matrix(1024, 4096, CONFIG0_PROBS, seed=0)
    n = m.bits.size
    for b, p in CONFIG0_PROBS.items():
        cnt = int((m.bits == b).sum())
        sigma = np.sqrt(n * p * (1 - p))
        assert abs(cnt - n * p) <= 4 * sigma, (b, cnt, n * p)
    # codes are in range and cover it
    for b in (1, 2, 4, 8):
        sel = np.repeat(m.bits == b, 64, axis=1)
        c = m.codes[sel]
        assert c.max() == (1 << b) - 1 and c.min() == 0
    s = m.scales.view(np.float16).astype(np.float64)
    assert s.min() >= 0.0099 and s.max() <= 0.0501


def test_stress_bit_maps():
    n, k = 256, 1024
    g = k // 64
    assert (stress_bits("a", n, k) == 1).all()
    assert (stress_bits("b", n, k) == 8).all()
    d = stress_bits("d", n, k)
    assert set(np.unique(d[: n // 2])) <= {4, 8} and (d[n // 2:] == 1).all()
    assert abs(d[: n // 2].astype(float).mean() - 6.0) < 0.2
    e = stress_bits("e", n, k)
    assert (e[:, : g // 4] == 8).all() and (e[:, g // 4:] == 1).all()
    m = gen_stress("e", n, k)
    assert O.storage_bytes(m.bits)["mean_bits"] == pytest.approx(2.75)


def test_generator_is_deterministic():
    a = gen_matrix(64, 256, CONFIG0_PROBS, seed=3)
    b = gen_matrix(64, 256, CONFIG0_PROBS, seed=3)
    c = gen_matrix(64, 256, CONFIG0_PROBS, seed=4)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.scales, b.scales)
    assert not np.array_equal(a.codes, c.codes)


# ---- decode-step glue ----

def test_rmsnorm_closed_form():
    for c in (0.5, -3.0, 1e-3):
        h = np.full(64, c)
        want = c / np.sqrt(c * c + O.RMS_EPS)
        np.testing.assert_allclose(O.rmsnorm(h), want, rtol=1e-15)
    rng = np.random.default_rng(0)
    h = rng.standard_normal(4096) * 7
    u = O.rmsnorm(h, eps=0.0)
    assert np.mean(u * u) == pytest.approx(1.0, rel=1e-13)
    assert np.all(np.sign(u) == np.sign(h))


def test_silu_identities():
    v = np.linspace(-20, 20, 4001)
    s = O.silu(v)
    np.testing.assert_allclose(s - O.silu(-v), v, atol=1e-12)   # silu(x) - silu(-x) = x
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(np.array([1.0])), 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)


def test_attention_pos0_equals_one_key_softmax():
    """A generic softmax attention over one cached key with GQA repeat = the shortcut."""
    rng = np.random.default_rng(2)
    H, Hkv, hd = 8, 2, 16
    q = rng.standard_normal((H, hd))
    k = rng.standard_normal((Hkv, 1, hd))        # one cached key per kv head
    v = rng.standard_normal((Hkv, 1, hd))
    kk = np.repeat(k, H // Hkv, axis=0)          # [H, 1, hd], kv head shared by H/Hkv queries
    vv = np.repeat(v, H // Hkv, axis=0)
    scores = np.einsum("hd,htd->ht", q, kk) / np.sqrt(hd)
    p = np.exp(scores - scores.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    out = np.einsum("ht,htd->hd", p, vv).reshape(-1)
    np.testing.assert_allclose(O.attention_pos0(v.reshape(-1), H, Hkv, hd), out, rtol=1e-15)


def _zero_scale_getter(tiny, keep):
    from synth import gen_model_matrix

    def get(layer, proj):
        m = gen_model_matrix(tiny, layer, proj, seed=0)
        s = m.scales if (layer, proj) in keep or proj in keep else np.zeros_like(m.scales)
        return m.codes, m.bits, s
    return get


def test_decode_step_residual_structure():
    """With every o and down projection zeroed, h stays x: logits = Whead bf16(rmsnorm(x))."""
    from synth import model_tiny, gen_model_matrix
    t = model_tiny()
    x = gen_x(t.d, seed=5)
    get = _zero_scale_getter(t, keep={"q", "k", "v", "gate", "up", "head"})
    logits = O.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, x)
    hm = gen_model_matrix(t, t.n_layers, "head", seed=0)
    u = O.f64_to_bf16_bits(O.rmsnorm(bf16_bits_to_f32(x).astype(np.float64)))
    assert np.array_equal(logits, O.gemv(hm.codes, hm.bits, hm.scales, u))


def test_decode_step_trace_chain():
    """The traced inputs are the bf16 glue of the traced outputs, step by step."""
    from synth import model_tiny, gen_model_matrix
    t = model_tiny()
    x = gen_x(t.d, seed=6)

    def get(layer, proj):
        m = gen_model_matrix(t, layer, proj, seed=0)
        return m.codes, m.bits, m.scales
    tr = []
    logits = O.decode_step(get, t.n_layers, t.n_heads, t.n_kv_heads, t.head_dim, x, trace=tr)
    assert len(tr) == 7 * t.n_layers + 1
    byname = {(l, p): (i, y) for l, p, i, y in tr}
    h = bf16_bits_to_f32(x).astype(np.float64)
    for layer in range(t.n_layers):
        i_q = byname[(layer, "q")][0]
        assert np.array_equal(i_q, O.f64_to_bf16_bits(O.rmsnorm(h)))
        v = byname[(layer, "v")][1]
        a = byname[(layer, "o")][0]
        grp = t.n_heads // t.n_kv_heads
        for head in range(t.n_heads):
            kv = head // grp
            seg = v[kv * t.head_dim:(kv + 1) * t.head_dim]
            assert np.array_equal(a[head * t.head_dim:(head + 1) * t.head_dim], O.f64_to_bf16_bits(seg))
        h = h + byname[(layer, "o")][1]
        m_in = byname[(layer, "down")][0]
        g, u = byname[(layer, "gate")][1], byname[(layer, "up")][1]
        assert np.array_equal(m_in, O.f64_to_bf16_bits(g / (1 + np.exp(-g)) * u))
        h = h + byname[(layer, "down")][1]
    assert np.array_equal(logits, byname[(t.n_layers, "head")][1])


# ---- stored fixtures written by tests/golden/make_golden.py (oracle only) ----

def _golden_files():
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json"))


@pytest.mark.parametrize("name", _golden_files())
def test_golden_fixture(name):
    with open(os.path.join(GOLDEN, name)) as f:
        fx = json.load(f)
    codes = np.array(fx["codes"], np.uint8)
    bits = np.array(fx["bits"], np.uint8)
    scales = np.array(fx["scales_f16_bits"], np.uint16)
    X = np.array(fx["x_bf16_bits"], np.uint16)
    Y = O.gemm(codes, bits, scales, X)
    want = np.array(fx["y"], np.float64)
    # fp64 sums may be ordered differently by another BLAS build: allow K ulps of sum|w x|
    W64 = O.dequant(codes, bits, scales).astype(np.float64)
    xs = bf16_bits_to_f32(X).astype(np.float64)
    bound = (np.abs(xs) @ np.abs(W64).T) * codes.shape[1] * 2.0 ** -52
    assert np.all(np.abs(Y - want) <= bound), fx["name"]
    W = O.dequant(codes, bits, scales)
    assert np.array_equal(W.view(np.uint32), np.array(fx["w_f32_bits"], np.uint32))
