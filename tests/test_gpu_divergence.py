"""The divergence measurement (GPU): a dense synthetic model quantized onto the VBQ grid at three
allocations (all 8-bit, the config-0 mix, all 1-bit) by the library's encoder, run through the
decode step, against the dense model's fp64 chain: KL divergence and argmax flips."""

import numpy as np
import pytest

from oracle import quant_oracle as Q
from oracle import vbq_oracle as O
from synth import CONFIG0_PROBS, gen_x, model_matrix_list, model_matrix_shape, model_tiny
from tests.gpu_util import dev_u16, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V(cuda_device):
    return lib()


def dense_weights(shape, seed):
    rng = np.random.default_rng(seed)
    W = {}
    for (layer, proj) in model_matrix_list(shape):
        n, k = model_matrix_shape(shape, proj)
        W[(layer, proj)] = (rng.standard_normal((n, k)) / np.sqrt(k)).astype(np.float32)
    return W


def divergence(V, shape, W, probs, xs, seed, with_oracle=False):
    import torch
    rng = np.random.default_rng(seed)
    handles = []
    packed = {}
    for (layer, proj) in model_matrix_list(shape):
        w = W[(layer, proj)]
        bits = rng.choice(list(probs.keys()), size=(w.shape[0], w.shape[1] // 64),
                          p=list(probs.values())).astype(np.uint8)
        codes, scales = V.vbq_quantize_rtn(w, bits)
        packed[(layer, proj)] = (codes, bits, scales)
        handles.append(V.Matrix(codes, bits, scales))
    desc = V.make_model_desc(shape.n_layers, shape.d, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                             shape.d_ff, shape.vocab, O.RMS_EPS)
    model = V.Model(desc, handles)
    got = []
    for x in xs:
        lg = torch.empty(shape.vocab, device="cuda")
        V.vbq_decode_step(model.handle, dev_u16(x), lg)
        torch.cuda.synchronize()
        got.append(lg.cpu().numpy().astype(np.float64))
    model.close()
    for h in handles:
        h.close()
    ref = [O.decode_step(None, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim, x,
                         dense=lambda layer, proj: W[(layer, proj)]) for x in xs]
    if not with_oracle:
        return Q.kl_and_flips(np.array(ref), np.array(got))
    # the oracle's fp64 chain over the same codes and scales: the VBQ side of the measurement without the GPU
    orc = [O.decode_step(lambda layer, proj: packed[(layer, proj)], shape.n_layers, shape.n_heads,
                         shape.n_kv_heads, shape.head_dim, x) for x in xs]
    return (Q.kl_and_flips(np.array(ref), np.array(got)), Q.kl_and_flips(np.array(ref), np.array(orc)),
            Q.kl_and_flips(np.array(orc), np.array(got)))


def test_divergence_grows_as_bits_shrink(V):
    shape = model_tiny()
    W = dense_weights(shape, seed=11)
    xs = [gen_x(shape.d, seed=100 + i) for i in range(8)]
    res = {}
    for name, probs in [("8bit", {8: 1.0}), ("config0", CONFIG0_PROBS), ("1bit", {1: 1.0})]:
        kl, flips = divergence(V, shape, W, probs, xs, seed=12)
        assert np.isfinite(kl).all() and (kl >= -1e-12).all()
        res[name] = (float(kl.mean()), float(flips.mean()))
    assert res["8bit"][0] < res["config0"][0] < res["1bit"][0], res
    assert res["8bit"][0] < 1e-3 and res["8bit"][1] == 0.0, res


def test_measured_divergence_is_the_oracles(V):
    """The KL and flips measured through the GPU step equal, within the step's own error, those of the
    oracle's fp64 chain over the same encodings; the GPU and oracle distributions are near-identical."""
    shape = model_tiny()
    W = dense_weights(shape, seed=11)
    xs = [gen_x(shape.d, seed=100 + i) for i in range(8)]
    for name, probs in [("8bit", {8: 1.0}), ("config0", CONFIG0_PROBS), ("1bit", {1: 1.0})]:
        (kl_g, fl_g), (kl_o, fl_o), (kl_og, _) = divergence(V, shape, W, probs, xs, seed=12, with_oracle=True)
        info = (name, kl_g.tolist(), kl_o.tolist(), kl_og.tolist(), fl_g.tolist(), fl_o.tolist())
        assert kl_og.max() <= 1e-3, info
        assert np.all(np.abs(kl_g - kl_o) <= 0.1 * kl_o + 1e-4), info
        assert int((fl_g != fl_o).sum()) <= 1, info
