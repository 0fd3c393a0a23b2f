"""GPU parity of the tcgen05 dequant->bf16 GEMM through the C ABI against the fp64
oracle: |Y - Y_ref| <= 8e-3 * sum_j |w^ x| (the oracle sums the exact decoded
weights times the bf16 activations the kernel received), plus exact special
cases: unit-vector rows give bf16(column), all-8 codes give zero."""
import numpy as np
import pytest

import synth
from gpu_helpers import bf16_round, within_tol

pytestmark = pytest.mark.gpu
TOL = 8e-3


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available()
    return t


@pytest.fixture(scope="module")
def q4():
    import bit_weight_quantized_03_b300 as m
    m.lib()
    return m


def _case(torch, oracle_mod, n, k, m, seed):
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=seed))
    xb = torch.from_numpy(synth.np_activations(m, k, seed=seed + 1)).to(torch.bfloat16)
    return W, xb


SHAPES = [(128, 256, 16), (77, 256, 1), (300, 3072, 129), (1000, 512, 300),
          (1280, 1280, 375), (3840, 1280, 64), (1280, 5120, 257), (130, 1024, 200),
          (256, 768, 513), (4096, 3072, 32)]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_gemm_matches_oracle(torch, q4, oracle_mod, n, k, m):
    W, xb = _case(torch, oracle_mod, n, k, m, seed=n + 3 * k + m)
    Y, S = oracle_mod.matmul(W, n, k, xb.float().numpy(), nthreads=oracle_mod.cpu_count())
    got = q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, xb.cuda()).cpu().numpy()
    ok, info = within_tol(got, Y, S, TOL)
    assert ok, info


# bf16 Y: even row strides take the epilogue's 4-byte stores of row pairs,
# odd strides 2-byte stores; n and m ragged so that an edge row pair and a tail
# token pair are cut.  Padding must stay untouched.
@pytest.mark.parametrize("n,k,m,pad", [(640, 1280, 100, 0), (334, 512, 37, 2),
                                       (129, 256, 3, 3), (333, 512, 37, 1),
                                       (333, 512, 37, 0), (200, 512, 65, 1)])
def test_gemm_bf16_output(torch, q4, oracle_mod, n, k, m, pad):
    W, xb = _case(torch, oracle_mod, n, k, m, seed=9 + n + pad)
    Y, S = oracle_mod.matmul(W, n, k, xb.float().numpy())
    Yd = torch.full((m, n + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, xb.cuda(), Y=Yd[:, :n])
    got = Yd.float().cpu().numpy()
    ok, info = within_tol(got[:, :n], Y, S, TOL)
    assert ok, info
    assert np.all(got[:, n:] == 7.0)


@pytest.mark.parametrize("n", [201, 202, 204])
def test_gemm_unit_rows_give_bf16_columns_in_bf16(torch, q4, oracle_mod, n):
    k = 256
    W, _ = _case(torch, oracle_mod, n, k, 1, seed=6)
    cols = oracle_mod.dequant_rows(W, n, k).T  # [k, n], exact fp32
    X = torch.eye(k, dtype=torch.bfloat16)
    got = q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, X.cuda(), y_dtype=torch.bfloat16)
    assert np.array_equal(got.float().cpu().numpy(), bf16_round(cols))


def test_gemm_unit_rows_give_bf16_columns(torch, q4, oracle_mod):
    n, k = 200, 512
    W, _ = _case(torch, oracle_mod, n, k, 1, seed=4)
    cols = oracle_mod.dequant_rows(W, n, k).T  # [k, n], exact fp32
    X = torch.eye(k, dtype=torch.bfloat16)
    got = q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, X.cuda()).cpu().numpy()
    assert np.array_equal(got, bf16_round(cols))


def test_gemm_all_eight_codes_give_zero(torch, q4):
    n, k, m = 256, 512, 40
    W = np.zeros((n, k // 32 * 18), np.uint8)
    blk = W.reshape(n, k // 32, 18)
    blk[:, :, 0:2] = np.frombuffer(np.float16(1.5).tobytes(), np.uint8)
    blk[:, :, 2:] = 0x88
    xb = torch.from_numpy(synth.np_activations(m, k, seed=2)).to(torch.bfloat16)
    got = q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, xb.cuda()).cpu().numpy()
    assert np.all(got == 0)


def test_gemm_strided_x_and_y(torch, q4, oracle_mod):
    n, k, m = 384, 768, 70
    W, xb = _case(torch, oracle_mod, n, k, m, seed=12)
    Y, S = oracle_mod.matmul(W, n, k, xb.float().numpy())
    Xs = torch.zeros((m, k + 64), dtype=torch.bfloat16, device="cuda")
    Xs[:, :k] = xb.cuda()
    Ys = torch.full((m, n + 12), 7.0, dtype=torch.float32, device="cuda")
    q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, Xs, Y=Ys)
    got = Ys.cpu().numpy()
    ok, info = within_tol(got[:, :n], Y, S, TOL)
    assert ok, info
    assert np.all(got[:, n:] == 7.0)


def test_gemm_deterministic(torch, q4, oracle_mod):
    n, k, m = 1280, 1280, 375
    W, xb = _case(torch, oracle_mod, n, k, m, seed=13)
    Wd, Xd = torch.from_numpy(W).cuda(), xb.cuda()
    a = q4.q4_gemm(Wd, n, k, Xd).cpu().numpy()
    b = q4.q4_gemm(Wd, n, k, Xd, flags=q4.FLAG_PDL).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gemm_m1_agrees_with_gemv(torch, q4, oracle_mod):
    n, k = 512, 1024
    W, xb = _case(torch, oracle_mod, n, k, 1, seed=14)
    Y, S = oracle_mod.matmul(W, n, k, xb.float().numpy())
    Wd = torch.from_numpy(W).cuda()
    yg = q4.q4_gemm(Wd, n, k, xb.cuda()).cpu().numpy()
    yv = q4.q4_gemv(Wd, n, k, xb.float().cuda()).cpu().numpy()
    assert np.all(np.abs(yg - yv) <= TOL * S)


@pytest.mark.parametrize("m", [1, 3, 5, 9, 16, 40, 200])
def test_linear_dispatch_matches_oracle(torch, q4, oracle_mod, m):
    n, k = 640, 3072
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=50 + m))
    x = synth.np_activations(m, k, seed=60 + m)
    Wd = torch.from_numpy(W).cuda()
    y = q4.q4_linear(Wd, n, k, torch.from_numpy(x).cuda()).cpu().numpy()
    gemv_path = m <= q4.q4_linear_crossover_m(n, k)
    xin = x if gemv_path else bf16_round(x)
    Y, S = oracle_mod.matmul(W, n, k, xin)
    ok, info = within_tol(y, Y, S, 1e-4 if gemv_path else TOL)
    assert ok, info


def test_gemm_split_k_leaves_workspace_zero(torch, q4, oracle_mod):
    """Small M splits K across CTAs; the partial tiles live in the workspace and
    must be cleared again, since GEMV calls share the same workspace."""
    n, k, m = 4096, 3072, 8
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=61))
    x = synth.np_activations(m, k, seed=62)
    ws = q4.Workspace()
    xb = torch.from_numpy(x).to(torch.bfloat16).cuda()
    y = q4.q4_gemm(torch.from_numpy(W).cuda(), n, k, xb, workspace=ws)
    torch.cuda.synchronize()
    assert q4.q4_gemm_workspace_bytes(n, k, m) > 0  # this shape does split K
    assert int(ws.buf.count_nonzero().item()) == 0
    Y, S = oracle_mod.matmul(W, n, k, xb.float().cpu().numpy())
    ok, info = within_tol(y.cpu().numpy(), Y, S, 8e-3)
    assert ok, info


def test_linear_refused_tensor_core_call_launches_nothing(torch, q4):
    """fp32 X with m above the GEMV batch and k % 256 != 0 cannot run on the
    tensor cores: the call is refused before the fp32 -> bf16 conversion is
    launched, so the shared workspace stays all zero for the next GEMV."""
    n, k, m = 64, 3104, 17
    W = torch.zeros((n, k // 32 * 18), dtype=torch.uint8, device="cuda")
    x = torch.ones((m, k), dtype=torch.float32, device="cuda")
    y = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    st = q4.lib().q4_linear(W.data_ptr(), n, k, x.data_ptr(), q4.F32, m, k, y.data_ptr(), n,
                            ws.data_ptr(), ws.numel(), None, 0, None)
    torch.cuda.synchronize()
    assert st == q4.ERR_UNSUPPORTED_SHAPE
    assert int(ws.count_nonzero().item()) == 0
