"""q4_gemv_q8 (the Q4 x Q8 integer path) against the oracle's Q4 x Q8 product
(per-32 int8 activations, exact integer block sums; READING stated in
oracle/q4_oracle.h): element-wise within 1e-4 of the block terms' magnitudes,
the Q8 error bound against the unquantized product, exact power-of-two
scaling, non-finite and zero blocks, at small ragged shapes and the decoder's
shapes."""
import numpy as np
import pytest

import synth
from gpu_helpers import within_tol

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    return t


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_03_b300 as m
    return m


def _case(oracle_mod, n, k, seed):
    W, rc, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=seed))
    assert rc == 0
    x = synth.np_activations(1, k, seed=seed + 1)[0]
    return W, x


@pytest.mark.parametrize("n,k", [(1, 32), (3, 64), (17, 96), (100, 256), (4096, 3072),
                                 (1024, 3072), (3072, 4096), (3072, 9216), (9216, 3072),
                                 (37, 12288)])
def test_gemv_q8_matches_oracle(torch, q4, oracle_mod, n, k):
    W, x = _case(oracle_mod, n, k, seed=n * 7 + k)
    y = q4.q4_gemv_q8(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda())
    got = y.cpu().numpy()
    Y, S = oracle_mod.matmul_q8(W, n, k, x)
    ok, info = within_tol(got, Y[0], S[0], TOL)
    assert ok, info
    # and the Q8 error model against the unquantized product
    _, d = oracle_mod.quantize_q8(x)
    Yx, Sx = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    w = np.abs(oracle_mod.dequant_rows(W, n, k).astype(np.float64))
    bound = w @ np.repeat(d.astype(np.float64) / 2, 32) + TOL * S[0] + 1e-12 * Sx[0]
    assert np.all(np.abs(got - Yx[0]) <= bound)


def test_gemv_q8_power_of_two_scaling_and_repeat(torch, q4, oracle_mod):
    n, k = 300, 1024
    W, x = _case(oracle_mod, n, k, seed=5)
    Wd = torch.from_numpy(W).cuda()
    a = q4.q4_gemv_q8(Wd, n, k, torch.from_numpy(x).cuda())
    b = q4.q4_gemv_q8(Wd, n, k, torch.from_numpy(x * np.float32(2.0 ** 7)).cuda())
    c = q4.q4_gemv_q8(Wd, n, k, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert torch.equal(b, a * 2.0 ** 7)
    assert torch.equal(a.view(torch.int32), c.view(torch.int32))


def test_gemv_q8_zero_and_nonfinite_blocks(torch, q4, oracle_mod):
    n, k = 40, 128
    W, x = _case(oracle_mod, n, k, seed=9)
    Wd = torch.from_numpy(W).cuda()
    z = q4.q4_gemv_q8(Wd, n, k, torch.zeros(k, device="cuda")).cpu().numpy()
    assert np.all(z == 0)
    x2 = x.copy()
    x2[70] = np.inf
    y = q4.q4_gemv_q8(Wd, n, k, torch.from_numpy(x2).cuda()).cpu().numpy()
    Y, _ = oracle_mod.matmul_q8(W, n, k, x2)
    assert np.all(np.isnan(Y[0])) and np.all(np.isnan(y))
