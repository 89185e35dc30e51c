"""The allocation-free decode step against vbq_decode_step and the oracle, through the C ABI (GPU).

vbq_decode_step_noalloc is for callers that may not allocate device memory, or
tie it to a model, at step time. It keeps the step's scratch in a static device
array instead of the model's workspace. This file is named so that pytest
collects it last: if it fails, a run that stops at the first failure has
already run every other test.
"""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import gen_model_matrix, gen_x, model_matrix_list, model_tiny
from tests.gpu_util import TOL, dev_u16, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _build(V, shape, seed):
    mats, handles = {}, []
    for (layer, proj) in model_matrix_list(shape):
        m = gen_model_matrix(shape, layer, proj, seed=seed)
        mats[(layer, proj)] = m
        handles.append(V.Matrix(m.codes, m.bits, m.scales))
    desc = V.make_model_desc(shape.n_layers, shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                             shape.d_ff, shape.vocab, O.RMS_EPS)
    return mats, handles, V.Model(desc, handles)


def test_noalloc_step_matches_decode_step_twice(V):
    import torch
    shape = model_tiny()
    mats, handles, model = _build(V, shape, seed=2)
    head = mats[(shape.n_layers, "head")]
    norms = O.row_norms(head.codes, head.bits, head.scales)
    get = lambda layer, proj: (mats[(layer, proj)].codes, mats[(layer, proj)].bits, mats[(layer, proj)].scales)
    for call, seed in enumerate((31, 32)):          # two calls in a row, different inputs
        x = gen_x(shape.d, seed=seed)
        xd = dev_u16(x)
        ref = torch.full((shape.vocab,), float("nan"), device="cuda")
        out = torch.full((shape.vocab,), float("nan"), device="cuda")
        V.vbq_decode_step(model.handle, xd, ref)
        V.vbq_decode_step_noalloc(model.handle, xd, out)
        torch.cuda.synchronize()
        r, o = ref.cpu().numpy(), out.cpu().numpy()
        assert np.isfinite(o).all(), call
        # The same kernel on the same inputs, and a step's sums do not depend on timing.
        assert np.array_equal(o, r), call
        # Against the oracle's fp64 chain from the same x (each bf16 rounding of a projection input
        # may differ by one ulp between the chains, so the bar is the end-to-end drift of the
        # decode tests, relative to the largest head row norm times sqrt(d)).
        chain = O.decode_step(get, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim, x)
        assert np.max(np.abs(o - chain)) / (np.max(norms) * np.sqrt(shape.d)) < 2e-2, call
    assert V.vbq_device_check() == 0
    model.close()
    for h in handles:
        h.close()


def test_noalloc_step_rejects_models_over_the_scratch_limit(V):
    import torch
    # The size check: a model that needs more words than the usable part of the
    # static array (lowered by a test hook) is refused and nothing is enqueued.
    shape = model_tiny()
    mats, handles, model = _build(V, shape, seed=3)
    x = dev_u16(gen_x(shape.d, seed=4))
    out = torch.zeros(shape.vocab, device="cuda")
    try:
        V.vbq_debug_set(V.VBQ_DEBUG_NOALLOC_WORDS, 1024)
        with pytest.raises(V.VbqError) as e:
            V.vbq_decode_step_noalloc(model.handle, x, out)
        assert e.value.status == 2 and "scratch" in e.value.detail
        torch.cuda.synchronize()
        assert (out.cpu().numpy() == 0).all()           # nothing was enqueued
    finally:
        V.vbq_debug_set(V.VBQ_DEBUG_NOALLOC_WORDS, 0)
    V.vbq_decode_step_noalloc(model.handle, x, out)   # the full array holds it
    torch.cuda.synchronize()
    assert np.isfinite(out.cpu().numpy()).all()
    model.close()
    for h in handles:
        h.close()
