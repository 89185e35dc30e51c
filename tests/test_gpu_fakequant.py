"""Fake quantization through the C ABI against the oracle (GPU): the mixture's forward and the
straight-through backward, every element, on ragged and edge inputs."""

import numpy as np
import pytest

from oracle import fakequant_oracle as F
from tests.gpu_util import lib
from tests.parity_bound import fakequant_tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("n,k,tau,zero_group", [(1, 64, 1.0, False), (37, 320, 0.5, True), (256, 4096, 2.0, False),
                                                (3, 128, 0.05, True)])
def test_fakequant_forward_backward(V, n, k, tau, zero_group):
    import torch
    rng = np.random.default_rng(n * 31 + k)
    W = (rng.standard_normal((n, k)) * 0.1).astype(np.float32)
    if zero_group:
        W[0, :64] = 0.0
    alpha = rng.standard_normal((n, k // 64, 4)).astype(np.float32)
    u = rng.uniform(0.01, 0.99, size=(n, k // 64, 4)).astype(np.float32)
    G = rng.standard_normal((n, k)).astype(np.float32)
    Wd, ad, ud, Gd = _dev(W), _dev(alpha), _dev(u), _dev(G)
    out = torch.full((n, k), float("nan"), device="cuda")
    dW = torch.full((n, k), float("nan"), device="cuda")
    da = torch.full((n, k // 64, 4), float("nan"), device="cuda")
    V.vbq_fakequant_forward(Wd, ad, ud, tau, n, k, out)
    V.vbq_fakequant_backward(Wd, ad, ud, tau, Gd, n, k, dW, da)
    torch.cuda.synchronize()
    ref = F.forward(W, alpha.astype(np.float64), u.astype(np.float64), tau)
    # the tolerances of the kernels' fp32 arithmetic (pinned on the CPU by test_fakequant_bound_cpu.py)
    tol, tol_a = fakequant_tolerances(W, tau, G)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), float((np.abs(got - ref) / tol).max())
    dW_ref, da_ref = F.backward(W, alpha.astype(np.float64), u.astype(np.float64), tau, G)
    assert np.array_equal(dW.cpu().numpy(), G)
    da_got = da.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(da_got - da_ref) <= tol_a), float((np.abs(da_got - da_ref) / tol_a).max())
