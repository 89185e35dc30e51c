"""Decode attention through the C ABI against the fp64 oracle (GPU).

* vbq_rope_append: q turned in place and the new k turned into the cache at
  pos, bit for bit (both sides rotate in fp64, round to fp32, then to bf16);
  v copied; every other cache position untouched.
* vbq_attention_decode: every output element within a bound of the kernel's
  fp32 arithmetic, on grouped and multi-head shapes, one span and many, a
  ragged last sub-chunk, kv_stride above T; repeated calls agree bit for bit.
"""

import numpy as np
import pytest

from oracle import attention_oracle as A
from oracle.vbq_oracle import bf16_bits_to_f64, f64_to_bf16_bits
from tests.gpu_util import dev_u16, lib
from tests.parity_bound import attention_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _bf16(rng, shape, scale=1.0):
    return f64_to_bf16_bits(rng.standard_normal(shape) * scale)


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("H,Hkv,d,pos", [(32, 8, 128, 0), (32, 8, 128, 1), (16, 16, 64, 37), (8, 1, 128, 4095)])
def test_rope_append(V, H, Hkv, d, pos):
    import torch
    rng = np.random.default_rng(H * 100 + pos)
    stride = 4096
    q = _bf16(rng, (H, d))
    kn, vn = _bf16(rng, (Hkv, d)), _bf16(rng, (Hkv, d))
    kc, vc = _bf16(rng, (Hkv, stride, d)), _bf16(rng, (Hkv, stride, d))
    qd, kd, vd = dev_u16(q), dev_u16(kc), dev_u16(vc)
    V.vbq_rope_append(qd, dev_u16(kn), dev_u16(vn), kd, vd, H, Hkv, d, stride, pos)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(qd), A.rope_bf16(q, pos))
    k_after, v_after = _u16(kd).reshape(Hkv, stride, d), _u16(vd).reshape(Hkv, stride, d)
    assert np.array_equal(k_after[:, pos], A.rope_bf16(kn, pos))
    assert np.array_equal(v_after[:, pos], vn)
    others = np.arange(stride) != pos
    assert np.array_equal(k_after[:, others], kc[:, others])
    assert np.array_equal(v_after[:, others], vc[:, others])


CASES = [  # H, Hkv, d, T, stride
    (32, 8, 128, 1, 8),
    (32, 8, 128, 200, 256),
    (32, 8, 128, 4096, 4096),
    (16, 16, 64, 300, 301),
    (12, 4, 64, 129, 130),
    (8, 1, 128, 65, 100),
    (32, 8, 128, 20000, 20001),
]


@pytest.mark.parametrize("H,Hkv,d,T,stride", CASES)
def test_attention_decode(V, H, Hkv, d, T, stride):
    import torch
    rng = np.random.default_rng(H + 7 * T + d)
    q = _bf16(rng, (H, d))
    kc, vc = _bf16(rng, (Hkv, stride, d)), _bf16(rng, (Hkv, stride, d))
    out = torch.full((H, d), float("nan"), device="cuda")
    qd, kd, vd = dev_u16(q), dev_u16(kc), dev_u16(vc)
    V.vbq_attention_decode(qd, kd, vd, H, Hkv, d, stride, T, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref, p = A.attention_decode(q, kc, vc, T)
    assert np.isfinite(got).all()
    bound = attention_bound(q, kc, vc, T, p)
    r = np.abs(got - ref) / bound
    assert r.max() <= 1.0, (float(r.max()), np.unravel_index(int(np.argmax(r)), r.shape))
    again = torch.full((H, d), float("nan"), device="cuda")
    V.vbq_attention_decode(qd, kd, vd, H, Hkv, d, stride, T, again)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().numpy(), out.cpu().numpy())


def test_rope_then_attention_chain(V):
    """A decode step's attention half: turn q and k at pos, append, attend over pos + 1 positions."""
    import torch
    rng = np.random.default_rng(99)
    H, Hkv, d, stride, pos = 32, 8, 128, 1024, 700
    q, kn, vn = _bf16(rng, (H, d)), _bf16(rng, (Hkv, d)), _bf16(rng, (Hkv, d))
    kc, vc = _bf16(rng, (Hkv, stride, d)), _bf16(rng, (Hkv, stride, d))
    qd, kd, vd = dev_u16(q), dev_u16(kc), dev_u16(vc)
    out = torch.full((H, d), float("nan"), device="cuda")
    V.vbq_rope_append(qd, dev_u16(kn), dev_u16(vn), kd, vd, H, Hkv, d, stride, pos)
    V.vbq_attention_decode(qd, kd, vd, H, Hkv, d, stride, pos + 1, out)
    torch.cuda.synchronize()
    qr = A.rope_bf16(q, pos)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, pos], vc2[:, pos] = A.rope_bf16(kn, pos), vn
    ref, p = A.attention_decode(qr, kc2, vc2, pos + 1)
    got = out.cpu().numpy().astype(np.float64)
    assert (np.abs(got - ref) / attention_bound(qr, kc2, vc2, pos + 1, p)).max() <= 1.0
