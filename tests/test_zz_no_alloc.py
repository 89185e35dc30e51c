"""The allocation-free decode step against vbq_decode_step, through the C ABI (GPU).

vbq_decode_step_noalloc is for callers that may not allocate device memory at
step time (for example while another component captures the stream into a CUDA
graph). It keeps its activations in a static device array instead of the model's
workspace. This file is named so that pytest
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
        # The parity bar of every GEMV test. The head's input is bf16(rmsnorm(h)), whose 2-norm is
        # sqrt(d), so a vector of ones stands in for it in the denominator.
        ones = O.f64_to_bf16_bits(np.ones(shape.d))
        # The same kernel on the same inputs; split tiles add their partial rows with fp32 atomic adds
        # in no fixed order, so the logits agree to the last bits only up to that order.
        assert O.normalized_error(o, r.astype(np.float64), norms, ones) <= TOL
    assert V.vbq_device_check() == 0
    model.close()
    for h in handles:
        h.close()


def test_noalloc_step_rejects_models_over_the_scratch_limit(V):
    import dataclasses
    import torch
    # 64 + 64 + 3*16384 ([q;k;v]) + 2*16384 ([gate;up]) = 82,048 floats > 65,536, with every
    # dimension within the decode kernel's limit of 16384 and every matrix small.
    big = dataclasses.replace(model_tiny(), name="wide", n_layers=1, d=64, n_heads=128, n_kv_heads=128,
                              head_dim=128, d_ff=16384, vocab=64)
    mats, handles, model = _build(V, big, seed=3)
    x = dev_u16(gen_x(big.d, seed=4))
    out = torch.zeros(big.vocab, device="cuda")
    with pytest.raises(V.VbqError) as e:
        V.vbq_decode_step_noalloc(model.handle, x, out)
    assert e.value.status == 2 and "scratch" in e.value.detail
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == 0).all()           # nothing was enqueued
    model.close()
    for h in handles:
        h.close()
