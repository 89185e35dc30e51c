"""Failure paths through the C ABI, without faulting the GPU (GPU).

* A wait that runs out: a test hook makes the decode step's flag waits look for
  a value no launch writes, with a short limit; the first wait gives up and
  records check code 3, the others give up at once, the launch completes, and
  vbq_device_check reports the code. The next normal step is clean.
* Out of memory: a host-side cap on the library's device allocations turns a
  pack into VBQ_ERR_OOM without exhausting the device.
* Rejected arguments: batch 0 and 65, and handles used on another device.
"""

import numpy as np
import pytest

from oracle import vbq_oracle as O
from synth import CONFIG0_PROBS, gen_matrix, gen_model_matrix, gen_x, model_matrix_list, model_tiny
from tests.gpu_util import dev_u16, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _tiny_model(V, seed):
    t = model_tiny()
    handles = []
    for (layer, proj) in model_matrix_list(t):
        m = gen_model_matrix(t, layer, proj, seed=seed)
        handles.append(V.Matrix(m.codes, m.bits, m.scales))
    desc = V.make_model_desc(t.n_layers, t.d, t.n_heads, t.n_kv_heads, t.head_dim, t.d_ff, t.vocab, O.RMS_EPS)
    return t, handles, V.Model(desc, handles)


@pytest.mark.parametrize("entry", ["vbq_decode_step", "vbq_decode_step_noalloc"])
def test_wait_that_runs_out_reports_code_3(V, entry):
    import torch
    t, handles, model = _tiny_model(V, seed=11)
    x = dev_u16(gen_x(t.d, seed=12))
    ref = torch.empty(t.vocab, device="cuda")
    V.vbq_decode_step(model.handle, x, ref)
    torch.cuda.synchronize()
    assert V.vbq_device_check() == 0
    out = torch.empty(t.vocab, device="cuda")
    try:
        V.vbq_debug_set(V.VBQ_DEBUG_WAIT_LIMIT, 100000)   # about 50 us
        V.vbq_debug_set(V.VBQ_DEBUG_NEVER_READY, 1)
        getattr(V, entry)(model.handle, x, out)
        torch.cuda.synchronize()                          # the launch completes
        with pytest.raises(V.VbqError) as e:
            V.vbq_device_check()
        assert e.value.status == 7 and "(code 3)" in e.value.detail
    finally:
        V.vbq_debug_set(V.VBQ_DEBUG_NEVER_READY, 0)
        V.vbq_debug_set(V.VBQ_DEBUG_WAIT_LIMIT, 0)
    # The step that gave up left the scratch as it found it: the next one is clean and exact.
    getattr(V, entry)(model.handle, x, out)
    torch.cuda.synchronize()
    assert V.vbq_device_check() == 0
    assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())
    model.close()
    for h in handles:
        h.close()


def test_allocation_cap_gives_oom(V):
    m = gen_matrix(2048, 2048, CONFIG0_PROBS, seed=13)
    try:
        V.vbq_debug_set(V.VBQ_DEBUG_ALLOC_CAP, 1 << 16)
        with pytest.raises(V.VbqError) as e:
            V.Matrix(m.codes, m.bits, m.scales)
        assert e.value.status == 6
    finally:
        V.vbq_debug_set(V.VBQ_DEBUG_ALLOC_CAP, 0)
    mat = V.Matrix(m.codes, m.bits, m.scales)         # without the cap it packs
    mat.close()
    assert V.vbq_device_check() == 0


@pytest.mark.parametrize("B", [0, 65, -1])
def test_smallbatch_rejects_batch_out_of_range(V, B):
    import torch
    m = gen_matrix(64, 256, CONFIG0_PROBS, seed=14)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    X = dev_u16(gen_x(256, seed=15, batch=65))
    Y = torch.full((65, 64), 7.0, device="cuda")
    with pytest.raises(V.VbqError) as e:
        V.vbq_gemm_smallbatch(mat.handle, X, B, Y)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert (Y.cpu().numpy() == 7.0).all()             # nothing was written
    mat.close()


def test_handles_from_another_device_are_rejected(V):
    import torch
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    m = gen_matrix(64, 256, CONFIG0_PROBS, seed=16)
    torch.cuda.set_device(1)
    mat = V.Matrix(m.codes, m.bits, m.scales)
    torch.cuda.set_device(0)
    x = dev_u16(gen_x(256, seed=17))
    y = torch.empty(64, device="cuda")
    with pytest.raises(V.VbqError) as e:
        V.vbq_gemv(mat.handle, x, y)
    assert e.value.status == 1
    torch.cuda.set_device(1)
    mat.close()
    torch.cuda.set_device(0)
