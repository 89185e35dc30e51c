"""The decode step at a position above 0 (GPU): each layer's rotary append and attention over its KV
cache between the projections, against the oracle under teacher forcing.

* At position 0 the context step gives vbq_decode_step's logits bit for bit.
* At positions 16 and 4095 (contexts 17 and 4096), with each layer's cache below pos filled with
  seeded values: every projection within the parity bar and the per-element bound for the GPU's
  own input; the new cache rows are the oracle's rotation of the GPU's k and v, bit for bit; each
  o input is the oracle's attention over the GPU's q and cache within the attention bound and one
  bf16 rounding; the RMSNorm and SwiGLU inputs as in the position-0 step; the logits near the fp64
  chain from the same input and caches.
"""

import numpy as np
import pytest

from oracle import attention_oracle as A
from oracle import vbq_oracle as O
from synth import gen_x, model_9b, model_tiny
from tests.gpu_util import bf16_ulp_diff, dev_u16
from tests.parity_bound import attention_bound
from tests.test_gpu_decode import Built, check_bounds, check_projections, glue_ulps, rmsnorm_input_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    from tests.gpu_util import lib
    return lib()


def _memcpy(dst, src, nbytes):
    from cuda.bindings import runtime as rt
    (err,) = rt.cudaMemcpy(dst, src, nbytes, rt.cudaMemcpyKind.cudaMemcpyDeviceToDevice)
    assert int(err) == 0, err


def fill_caches(V, b, pos, seed):
    """Seeded bf16 keys and values at positions < pos of every layer's caches (0 at and above pos)."""
    import torch
    s = b.shape
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for layer in range(s.n_layers):
        kp, vp, stride = V.vbq_model_kv_cache(b.model.handle, layer)
        for ptr in (kp, vp):
            t = (torch.randn(s.n_kv_heads, stride, s.head_dim, device="cuda", generator=g) * 2.0).to(torch.bfloat16)
            t[:, pos:, :] = 0
            _memcpy(ptr, t.data_ptr(), t.numel() * 2)
    torch.cuda.synchronize()


def read_cache(V, b, layer):
    import torch
    s = b.shape
    kp, vp, stride = V.vbq_model_kv_cache(b.model.handle, layer)
    out = []
    for ptr in (kp, vp):
        t = torch.empty(s.n_kv_heads, stride, s.head_dim, dtype=torch.int16, device="cuda")
        _memcpy(t.data_ptr(), ptr, t.numel() * 2)
        torch.cuda.synchronize()
        out.append(t.cpu().numpy().view(np.uint16))
    return out


def run_step_at(V, b, x, pos, trace=False):
    import torch
    V.vbq_model_set_trace(b.model.handle, trace)
    logits = torch.full((b.shape.vocab,), float("nan"), device="cuda")
    V.vbq_decode_step_at(b.model.handle, dev_u16(x), pos, logits)
    torch.cuda.synchronize()
    out = logits.cpu().numpy()
    if not trace:
        return out, None
    from synth import model_matrix_shape
    n = len(b.order)
    in_off, out_off, it, ot = V.vbq_model_trace_info(b.model.handle, n)
    tin, tout = V.vbq_model_read_trace(b.model.handle, it, ot)
    per = {}
    for i, (layer, proj) in enumerate(b.order):
        N, K = model_matrix_shape(b.shape, proj)
        per[(layer, proj)] = (tin[in_off[i]:in_off[i] + K], tout[out_off[i]:out_off[i] + N])
    return out, per


def check_attention_glue(V, b, per, x, pos, caches_before):
    """The glue of a step at pos: the cache rows written at pos, each o input against the oracle's
    attention over the GPU's own q, k, v and cache, then RMSNorm and SwiGLU inputs as at position 0."""
    s = b.shape
    h = O.bf16_bits_to_f64(x)
    err_h = np.zeros_like(h)
    near, total, o_off = 0, 0, 0

    def residual(h, err_h, v):
        v = v.astype(np.float64)
        new = h + v
        return new, err_h + 2.0 ** -20 * (np.abs(new) + np.abs(h) + np.abs(v)) + 2.0 ** -24 * err_h

    for layer in range(s.n_layers):
        near += rmsnorm_input_ok(per[(layer, "q")][0], h, err_h)
        total += h.size
        q = per[(layer, "q")][1].astype(np.float64)
        k = per[(layer, "k")][1].astype(np.float64)
        v = per[(layer, "v")][1].astype(np.float64)
        kc, vc = caches_before[layer]
        out, rows = A.step_attention(q, k, v, kc, vc, pos)
        kc_after, vc_after = read_cache(V, b, layer)
        assert np.array_equal(kc_after[:, pos], rows[0]) and np.array_equal(vc_after[:, pos], rows[1])
        assert np.array_equal(kc_after[:, :pos], kc[:, :pos]) and np.array_equal(vc_after[:, :pos], vc[:, :pos])
        # bound of the GPU's fp32 attention, then one bf16 rounding of each side
        qb = A.rope_bf16(O.f64_to_bf16_bits(q).reshape(s.n_heads, s.head_dim), pos)
        kc2, vc2 = kc.copy(), vc.copy()
        kc2[:, pos], vc2[:, pos] = rows[0], rows[1]
        _, p = A.attention_decode(qb, kc2, vc2, pos + 1)
        bound = attention_bound(qb, kc2, vc2, pos + 1, p).reshape(-1)
        got = O.bf16_bits_to_f64(per[(layer, "o")][0])
        _, e = np.frexp(np.maximum(np.abs(out), np.abs(got)))
        ulp = np.ldexp(1.0, np.maximum(e, -125) - 8)
        bad = np.abs(got - out) > bound + ulp
        assert not bad.any(), (layer, np.flatnonzero(bad)[:8])
        ref_bits = O.f64_to_bf16_bits(out)
        d = bf16_ulp_diff(per[(layer, "o")][0], ref_bits)
        near += int((d > 0).sum())
        total += d.size
        h, err_h = residual(h, err_h, per[(layer, "o")][1])
        near += rmsnorm_input_ok(per[(layer, "gate")][0], h, err_h)
        total += h.size
        g = per[(layer, "gate")][1].astype(np.float64)
        up = per[(layer, "up")][1].astype(np.float64)
        mm = O.f64_to_bf16_bits(O.silu(g) * up)
        dd = glue_ulps(per[(layer, "down")][0], mm)
        assert dd.max() <= 1
        near += int((dd > 0).sum())
        total += dd.size
        h, err_h = residual(h, err_h, per[(layer, "down")][1])
    near += rmsnorm_input_ok(per[(s.n_layers, "head")][0], h, err_h)
    total += h.size
    assert near <= max(8, total // 200), (near, total)


def test_context_step_at_position_zero_is_the_step(V):
    import torch
    b = Built(V, model_tiny(), seed=5)
    V.vbq_model_set_context(b.model.handle, 16)
    fill_caches(V, b, 16, seed=1)  # whatever the cache holds, position 0 attends to itself only
    x = gen_x(b.shape.d, seed=7)
    ref = torch.empty(b.shape.vocab, device="cuda")
    V.vbq_decode_step(b.model.handle, dev_u16(x), ref)
    got, _ = run_step_at(V, b, x, 0)
    assert np.array_equal(got, ref.cpu().numpy())
    assert V.vbq_device_check() == 0
    b.close()


@pytest.mark.parametrize("pos", [16, 4095])
def test_context_step_teacher_forced(V, pos):
    b = Built(V, model_tiny(), seed=6)
    V.vbq_model_set_context(b.model.handle, 4096)
    fill_caches(V, b, pos, seed=2)
    before = [read_cache(V, b, layer) for layer in range(b.shape.n_layers)]
    x = gen_x(b.shape.d, seed=8)
    logits, per = run_step_at(V, b, x, pos, trace=True)
    assert np.isfinite(logits).all()
    assert np.array_equal(per[(b.shape.n_layers, "head")][1], logits)
    check_projections(b, per)
    check_bounds(b, per, range(b.shape.n_layers))
    check_attention_glue(V, b, per, x, pos, before)
    # end to end (information): the fp64 chain from the same x and caches
    def attend(layer, q, k, v):
        kc, vc = before[layer]
        return A.step_attention(q, k, v, kc, vc, pos)[0]
    ref = O.decode_step(b.get, b.shape.n_layers, b.shape.n_heads, b.shape.n_kv_heads, b.shape.head_dim, x,
                        attend=attend)
    hm = b.get(b.shape.n_layers, "head")
    drift = np.max(np.abs(logits - ref)) / (np.max(O.row_norms(*hm)) * np.sqrt(b.shape.d))
    assert drift < 2e-2
    # the same step again: bit for bit (the cache row at pos is rewritten with the same values)
    again, _ = run_step_at(V, b, x, pos)
    assert np.array_equal(again, logits)
    assert V.vbq_device_check() == 0
    b.close()


def test_9b_context_4096_sampled(V):
    """The 9B-shaped step at context 4096: sampled rows of every projection, the first layer's
    projections on every row, the new cache rows and every o input of every layer."""
    b = Built(V, model_9b(), keep_inputs=False)
    pos = 4095
    V.vbq_model_set_context(b.model.handle, 4096)
    fill_caches(V, b, pos, seed=3)
    before = [read_cache(V, b, layer) for layer in range(b.shape.n_layers)]
    x = gen_x(b.shape.d, seed=9)
    logits, per = run_step_at(V, b, x, pos, trace=True)
    assert np.isfinite(logits).all()
    check_projections(b, per, rows_per_proj=6)
    check_bounds(b, per, [0])
    check_attention_glue(V, b, per, x, pos, before)
    assert V.vbq_device_check() == 0
    b.close()
