"""GPU decode step against the oracle: every projection under teacher forcing, the glue, and the logits."""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import PROJS, gen_model_matrix, gen_x, model_1b, model_9b, model_matrix_list, model_matrix_shape, model_tiny
from tests import parity_bound as PB
from tests.gpu_util import TOL, bf16_ulp_diff, dev_u16, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


class Built:
    def __init__(self, V, shape, seed=0, keep_inputs=True):
        self.shape = shape
        self.seed = seed
        self.mats = {}
        self.handles = []
        for (layer, proj) in model_matrix_list(shape):
            m = gen_model_matrix(shape, layer, proj, seed=seed)
            if keep_inputs:
                self.mats[(layer, proj)] = m
            self.handles.append(V.Matrix(m.codes, m.bits, m.scales))
        self.desc = V.make_model_desc(shape.n_layers, shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                                      shape.d_ff, shape.vocab, O.RMS_EPS)
        self.model = V.Model(self.desc, self.handles)
        self.order = model_matrix_list(shape)

    def get(self, layer, proj):
        m = self.mats.get((layer, proj))
        if m is None:  # not kept: draw it again (the generator is deterministic)
            m = gen_model_matrix(self.shape, layer, proj, seed=self.seed)
        return m.codes, m.bits, m.scales

    def close(self):
        self.model.close()
        for h in self.handles:
            h.close()


def run_step(V, b, x, trace=False):
    import torch
    V.vbq_model_set_trace(b.model.handle, trace)
    logits = torch.full((b.shape.vocab,), float("nan"), device="cuda")
    V.vbq_decode_step(b.model.handle, dev_u16(x), logits)
    torch.cuda.synchronize()
    out = logits.cpu().numpy()
    if not trace:
        return out, None
    n = len(b.order)
    in_off, out_off, it, ot = V.vbq_model_trace_info(b.model.handle, n)
    tin, tout = V.vbq_model_read_trace(b.model.handle, it, ot)
    per = {}
    for i, (layer, proj) in enumerate(b.order):
        N, K = model_matrix_shape(b.shape, proj)
        per[(layer, proj)] = (tin[in_off[i]:in_off[i] + K], tout[out_off[i]:out_off[i] + N])
    return out, per


def check_projections(b, per, rows_per_proj=None, seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for key, (xin, yout) in per.items():
        codes, bits, scales = b.get(*key)
        rows = None
        if rows_per_proj is not None and codes.shape[0] > rows_per_proj:
            rows = np.unique(np.r_[0, codes.shape[0] - 1, rng.integers(0, codes.shape[0], rows_per_proj)])
            codes, bits, scales, yout = codes[rows], bits[rows], scales[rows], yout[rows]
        ref = O.gemv(codes, bits, scales, xin)
        err = O.normalized_error(yout, ref, O.row_norms(codes, bits, scales), xin)
        assert err <= TOL, (key, err)
        worst = max(worst, err)
    return worst


ITEMS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def check_bounds(b, per, layers, head=True):
    """Every output row of the given layers' projections (and the head) within the per-element bound of
    the CUDA-core arithmetic, for the GPU's own traced input. Each CTA's fixed-point unit is at most the
    one from the whole input's max |x| and the item's L1 bound, and its 64-bit sums carry 32 more bits."""
    groups = [(layer, g) for layer in layers for g in ITEMS]
    if head:
        groups.append((b.shape.n_layers, ("head",)))
    worst = 0.0
    for layer, group in groups:
        mats = {p: b.get(layer, p) for p in group}
        l1 = max(PB.max_row_l1(*mats[p]) for p in group)
        x = per[(layer, group[0])][0]
        F = PB.fixed_exponent(l1, float(np.abs(O.bf16_bits_to_f64(x)).max()))
        for p in group:
            y = per[(layer, p)][1]
            ref = O.gemv(*mats[p], x)
            bound = PB.cuda_core_bound(*mats[p], x, F, slack_units=2.0 ** -8)
            worst = max(worst, PB.check_within(y, ref, bound))
    return worst


UNDERFLOW = 2.0 ** -100


def glue_ulps(gpu_bits, ref_bits):
    """bf16 ulp distance, with both-negligible pairs counted as equal.

    silu(g) = g / (1 + exp(-g)) in fp32 returns 0 once exp(-g) overflows
    (g < -88.7), where the exact fp64 value is below |g| e^g |up| < 1e-30 and
    still lands on some bf16 subnormal or tiny normal. Pairs whose magnitudes
    are both below 2^-100 are therefore not compared in ulps.
    """
    d = bf16_ulp_diff(gpu_bits, ref_bits)
    a = np.abs(O.bf16_bits_to_f64(gpu_bits))
    r = np.abs(O.bf16_bits_to_f64(ref_bits))
    return np.where((a <= UNDERFLOW) & (r <= UNDERFLOW), 0, d)


def rmsnorm_input_ok(gpu_bits, h, err_h):
    """The GPU's bf16(rmsnorm(h)) against the fp64 value, within rounding.

    The GPU keeps h in fp32, and each residual add rounds once, so its h is off
    by at most err_h per element (tracked by the caller). Where h nearly cancels,
    that absolute error is a large relative one, so the bound is absolute:
    one bf16 ulp of the exact value, plus err_h scaled by 1/rms, plus 2^-20
    relative for the fp32 sum of squares.
    """
    ref = O.rmsnorm(h)
    inv = 1.0 / np.sqrt(np.mean(h * h) + O.RMS_EPS)
    got = O.bf16_bits_to_f64(gpu_bits)
    _, e = np.frexp(ref)
    ulp = np.ldexp(1.0, np.maximum(e, -125) - 8)
    tol = ulp + err_h * inv + 2.0 ** -20 * np.abs(ref)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.flatnonzero(bad)[:8], got[bad][:8], ref[bad][:8])
    return int((O.f64_to_bf16_bits(ref) != gpu_bits).sum())


def check_glue(b, per, x):
    """Each projection input is the oracle's glue applied to the GPU's own earlier outputs."""
    s = b.shape
    h = O.bf16_bits_to_f64(x)
    err_h = np.zeros_like(h)      # bound on |h_gpu - h| from the fp32 residual adds
    near = 0
    total = 0

    def residual(h, err_h, v):
        # The kernel adds each projection's fp32 output onto the fp32 h once:
        # allow one rounding of the output and of h per add (generously).
        v = v.astype(np.float64)
        new = h + v
        return new, err_h + 2.0 ** -20 * (np.abs(new) + np.abs(h) + np.abs(v)) + 2.0 ** -24 * err_h

    for layer in range(s.n_layers):
        near += rmsnorm_input_ok(per[(layer, "q")][0], h, err_h)
        total += h.size
        v = per[(layer, "v")][1].astype(np.float64)
        a = O.f64_to_bf16_bits(O.attention_pos0(v, s.n_heads, s.n_kv_heads, s.head_dim))
        assert np.array_equal(per[(layer, "o")][0], a)  # same fp32 v, same rounding
        h, err_h = residual(h, err_h, per[(layer, "o")][1])
        near += rmsnorm_input_ok(per[(layer, "gate")][0], h, err_h)
        total += h.size
        g = per[(layer, "gate")][1].astype(np.float64)
        up = per[(layer, "up")][1].astype(np.float64)
        mm = O.f64_to_bf16_bits(O.silu(g) * up)
        d = glue_ulps(per[(layer, "down")][0], mm)
        assert d.max() <= 1
        near += int((d > 0).sum())
        total += d.size
        h, err_h = residual(h, err_h, per[(layer, "down")][1])
    near += rmsnorm_input_ok(per[(s.n_layers, "head")][0], h, err_h)
    total += h.size
    # Rounding differences come only from fp32-vs-fp64 values that sit near a bf16 rounding tie
    assert near <= max(8, total // 200), (near, total)


def test_tiny_decode_step_teacher_forced(V):
    b = Built(V, model_tiny())
    x = gen_x(b.shape.d, seed=3)
    logits, per = run_step(V, b, x, trace=True)
    assert np.isfinite(logits).all()
    assert np.array_equal(per[(b.shape.n_layers, "head")][1], logits)
    check_projections(b, per)
    check_bounds(b, per, range(b.shape.n_layers))
    check_glue(b, per, x)
    # end to end (information): the fp64 chain from the same x
    ref = O.decode_step(b.get, b.shape.n_layers, b.shape.n_heads, b.shape.n_kv_heads, b.shape.head_dim, x)
    hm = b.get(b.shape.n_layers, "head")
    drift = np.max(np.abs(logits - ref)) / (np.max(O.row_norms(*hm)) * np.sqrt(b.shape.d))
    assert drift < 2e-2
    b.close()


def test_decode_step_repeatable_and_host_path(V):
    """Steps on the same input give the same logits bit for bit: every sum of a step is an integer
    add or a float reduction in a fixed order, whatever the timing of the CTAs."""
    import torch
    b = Built(V, model_tiny(), seed=1)
    x = gen_x(b.shape.d, seed=4)
    l1, _ = run_step(V, b, x)
    assert np.isfinite(l1).all()
    l2, _ = run_step(V, b, x)          # new device buffers
    assert np.array_equal(l2, l1)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    lh = torch.empty(b.shape.vocab, dtype=torch.float32).pin_memory()
    V.vbq_decode_step_host(b.model.handle, xh, lh)
    assert np.array_equal(lh.numpy(), l1)
    # trace off and on give the same logits
    l3, _ = run_step(V, b, x, trace=True)
    assert np.array_equal(l3, l1)
    b.close()


def test_model_shape_mismatch_rejected(V):
    t = model_tiny()
    mats = []
    for (layer, proj) in model_matrix_list(t):
        m = gen_model_matrix(t, layer, proj, seed=0)
        mats.append(V.Matrix(m.codes, m.bits, m.scales))
    mats[3], mats[4] = mats[4], mats[3]   # o and gate swapped
    desc = V.make_model_desc(t.n_layers, t.d, t.n_heads, t.n_kv_heads, t.head_dim, t.d_ff, t.vocab)
    with pytest.raises(V.VbqError) as e:
        V.Model(desc, mats)
    assert e.value.status == 2
    for m in mats:
        m.close()


def test_1b_decode_step_sampled(V):
    b = Built(V, model_1b())
    x = gen_x(b.shape.d, seed=5)
    logits, per = run_step(V, b, x, trace=True)
    assert np.isfinite(logits).all()
    check_projections(b, per, rows_per_proj=24)
    check_bounds(b, per, [0, b.shape.n_layers - 1])
    check_glue(b, per, x)
    b.close()
    assert V.vbq_device_check() == 0


def test_9b_decode_step_sampled(V):
    """The full-size 9B-shaped step, in the launch configuration the bench times: every projection under
    teacher forcing on sampled rows (the first, the last and random ones), and the glue between them."""
    b = Built(V, model_9b(), keep_inputs=False)
    x = gen_x(b.shape.d, seed=6)
    logits, per = run_step(V, b, x, trace=True)
    assert np.isfinite(logits).all()
    check_projections(b, per, rows_per_proj=6)
    check_bounds(b, per, [0])        # a full layer (every row of its seven projections) and the head
    check_glue(b, per, x)
    b.close()
    assert V.vbq_device_check() == 0


def test_decode_step_zero_input(V):
    """x = 0: every RMSNorm input is 0, so every projection input and output and the logits are 0."""
    b = Built(V, model_tiny(), seed=2)
    logits, per = run_step(V, b, np.zeros(b.shape.d, np.uint16), trace=True)
    assert np.array_equal(logits, np.zeros_like(logits))
    for key, (xin, yout) in per.items():
        assert not xin.any() and not yout.any(), key
    b.close()
