"""The encoder-to-decoder bridge ("Conv with 4x downsampling -> adapter (3072
dimensions)", GeekNews es.news.hada.io/topic?id=26595, "Arquitectura") through
q4_gemm, with the shapes the stack assumes (synth.ADAPTER_MATS): each of the
three products element-wise against the oracle's fp64 product on the bf16
input that product read, on sampled output frames."""
import numpy as np
import pytest

import synth
from gpu_helpers import within_tol

pytestmark = pytest.mark.gpu
GEMM_TOL = 8e-3


@pytest.fixture(scope="module")
def torch():
    import torch as t
    return t


def test_adapter_stack_each_product_vs_oracle(torch, oracle_mod):
    from bit_weight_quantized_03_b300.stacks import AdapterStack
    ad = AdapterStack()
    X = synth.torch_activations(ad.frames, 1280, seed=synth.activation_seed(6000),
                                dtype=torch.bfloat16)
    out = ad.forward(X)
    torch.cuda.synchronize()
    assert out.shape == (375, 3072)
    inp = X.reshape(ad.m, 5120).float().cpu().numpy()
    rows = np.unique(np.concatenate([[0, ad.m - 1],
                                     np.random.default_rng(6).integers(0, ad.m, 30)]))
    th = oracle_mod.cpu_count()
    for idx, ((name, n, k), Y) in enumerate(zip(ad.mats, ad.Y)):
        w = synth.torch_weights(n, k, seed=synth.seed_for(6, 0, idx)).cpu().numpy()
        W, rc, _ = oracle_mod.quantize(w)
        assert rc == 0
        assert np.array_equal(ad.W[idx].cpu().numpy(), W)  # the GPU quantizer's blocks
        Yr, Sr = oracle_mod.matmul(W, n, k, inp[rows], nthreads=th)
        got = Y.float().cpu().numpy()
        ok, info = within_tol(got[rows], Yr, Sr, GEMM_TOL)
        assert ok, (name, info)
        inp = got


def test_adapter_rejects_frames_not_divisible_by_four(torch):
    from bit_weight_quantized_03_b300.stacks import AdapterStack
    with pytest.raises(ValueError):
        AdapterStack(encoder_frames=1501)
