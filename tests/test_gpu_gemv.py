"""GPU parity of the fp32 dequant-GEMV through the C ABI against the fp64 oracle:
|y - y_ref| <= 1e-4 * sum_j |w^ x| for every output, plus the exact special
cases (unit vectors, all-8 codes, power-of-two scaling) and run-to-run
determinism of the split-K reduction."""
import numpy as np
import pytest

import synth
from gpu_helpers import within_tol

pytestmark = pytest.mark.gpu
TOL = 1e-4


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


def _case(oracle_mod, n, k, m, seed):
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=seed))
    x = synth.np_activations(m, k, seed=seed + 1)
    return W, x


def _gemv(torch, q4, W, n, k, x, **kw):
    y = q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda(), **kw)
    return y.cpu().numpy()


# several tiles and ragged tails: n not a multiple of 32, k a multiple of 256
# (streamed kernel) or only of 32 (generic kernel)
# (several rows of x: launches of up to 4 rows of the batched tile kernel, 3
# where 4 rows of x do not fit in shared memory (k = 9216, 10240), and a single
# leftover row on the batch-1 kernel)
SHAPES = [(1, 32, 1), (3, 288, 2), (4095, 256, 1), (33, 512, 3), (4096, 3072, 1),
          (1000, 3072, 4), (257, 9216, 1), (3072, 4096, 2), (96, 256, 16), (130, 1280, 8),
          (64, 2304, 5), (1, 9216, 1), (2, 256, 9), (1, 256, 2), (4096, 3072, 3),
          (6144, 3072, 4), (257, 9216, 4), (100, 10240, 4), (3072, 9216, 7),
          # x too wide for the tile kernels' shared memory: the streamed kernel
          (64, 20480, 3), (33, 24576, 2), (40, 24576, 1)]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_gemv_matches_oracle(torch, q4, oracle_mod, n, k, m):
    W, x = _case(oracle_mod, n, k, m, seed=n + k + m)
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    y = _gemv(torch, q4, W, n, k, x)
    ok, info = within_tol(y, Y, S, TOL)
    assert ok, info


# Batch-1 calls with the PDL flag take the chain shape of the batch-1 kernel
# (8 warps per CTA, ring filled before the wait on the previous kernel) while
# its shared memory lets two CTAs share an SM (k up to 9216 here); k = 10240
# does not fit and falls back to the solo shape.
PDL_SHAPES = [(1, 256, 1), (4095, 256, 1), (4096, 3072, 1), (6144, 3072, 1), (257, 9216, 1),
              (3072, 9216, 1), (100, 10240, 1)]


@pytest.mark.parametrize("n,k,m", PDL_SHAPES)
def test_gemv_pdl_shape_matches_oracle(torch, q4, oracle_mod, n, k, m):
    W, x = _case(oracle_mod, n, k, m, seed=3 * n + k)
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    ws = q4.Workspace()
    ys = [_gemv(torch, q4, W, n, k, x, flags=q4.FLAG_PDL, workspace=ws) for _ in range(2)]
    ok, info = within_tol(ys[0], Y, S, TOL)
    assert ok, info
    assert np.array_equal(ys[1].view(np.uint32), ys[0].view(np.uint32))  # deterministic
    torch.cuda.synchronize()
    assert int(ws.buf.count_nonzero().item()) == 0


def test_gemv_strided_x_and_y(torch, q4, oracle_mod):
    n, k, m = 300, 1024, 3
    W, x = _case(oracle_mod, n, k, m, seed=5)
    Y, S = oracle_mod.matmul(W, n, k, x)
    xs = torch.zeros((m, k + 64), dtype=torch.float32, device="cuda")
    xs[:, :k] = torch.from_numpy(x).cuda()
    ys = torch.full((m, n + 7), 12345.0, dtype=torch.float32, device="cuda")
    q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, xs, y=ys)
    got = ys.cpu().numpy()
    ok, info = within_tol(got[:, :n], Y, S, TOL)
    assert ok, info
    assert np.all(got[:, n:] == 12345.0)  # nothing written past n


def test_gemv_unit_vectors_give_columns(torch, q4, oracle_mod):
    n, k = 77, 512
    W, _ = _case(oracle_mod, n, k, 1, seed=8)
    cols = oracle_mod.dequant_rows(W, n, k).T  # [k, n]
    for j0 in range(0, k, 16):  # 16 unit vectors per call
        x = np.zeros((16, k), np.float32)
        x[np.arange(16), j0 + np.arange(16)] = 1.0
        y = _gemv(torch, q4, W, n, k, x)
        assert np.array_equal(y, cols[j0:j0 + 16])  # exact (+0 and -0 compare equal)


def test_gemv_all_eight_codes_give_zero(torch, q4):
    n, k = 70, 768
    W = np.zeros((n, k // 32 * 18), np.uint8)
    blk = W.reshape(n, k // 32, 18)
    blk[:, :, 0:2] = np.frombuffer(np.float16(-2.75).tobytes(), np.uint8)
    blk[:, :, 2:] = 0x88
    x = synth.np_activations(2, k, seed=3)
    y = _gemv(torch, q4, W, n, k, x)
    assert np.all(y == 0)


def test_gemv_power_of_two_scaling_is_exact(torch, q4, oracle_mod):
    n, k = 129, 1024
    W, x = _case(oracle_mod, n, k, 1, seed=21)
    y1 = _gemv(torch, q4, W, n, k, x)
    y2 = _gemv(torch, q4, W, n, k, x * np.float32(2.0 ** -6))
    assert np.array_equal(y2, y1 * np.float32(2.0 ** -6))


def test_gemv_deterministic_and_pdl(torch, q4, oracle_mod):
    n, k, m = 4096, 3072, 2
    W, x = _case(oracle_mod, n, k, m, seed=30)
    Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
    ys = [q4.q4_gemv(Wd, n, k, xd).cpu().numpy() for _ in range(3)]
    ys.append(q4.q4_gemv(Wd, n, k, xd, flags=q4.FLAG_PDL).cpu().numpy())
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint32), ys[0].view(np.uint32))


def test_gemv_workspace_left_zeroed(torch, q4, oracle_mod):
    n, k, m = 1000, 3072, 1
    W, x = _case(oracle_mod, n, k, m, seed=31)
    ws = q4.Workspace()
    q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda(), workspace=ws)
    torch.cuda.synchronize()
    nb = q4.q4_gemv_workspace_bytes(n, k, m)
    assert nb > 0
    cnt_bytes = ((n + 31) // 32 * 4 + 255) // 256 * 256
    assert int(ws.buf[:cnt_bytes].count_nonzero().item()) == 0


@pytest.mark.parametrize("pdl", [False, True])
def test_gemv_bounded_wait_reports_timeout(torch, q4, oracle_mod, pdl):
    """A wait that nothing completes (test flag) ends with Q4_ERR_TIMEOUT in the
    status word after about a second; the context stays usable.  With the PDL
    flag the batch-1 kernel runs in its chain shape."""
    n, k = 64, 512
    W, x = _case(oracle_mod, n, k, 1, seed=40)
    ws = q4.Workspace()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = q4.FLAG_TEST_STALL | (q4.FLAG_PDL if pdl else 0)
    q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda(), workspace=ws,
               status=st, flags=flags)
    torch.cuda.synchronize()
    assert int(st.item()) == q4.ERR_TIMEOUT
    ws.reset()
    Y, S = oracle_mod.matmul(W, n, k, x)
    y = q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda(), workspace=ws)
    ok, info = within_tol(y.cpu().numpy(), Y, S, TOL)
    assert ok, info


def test_gemv_workspace_shared_across_shapes(torch, q4, oracle_mod):
    """One workspace used by calls of different shapes in a row: each call must
    leave all of it zero so the next shape's counters start from zero."""
    ws = q4.Workspace()
    for (n, k, m) in [(33, 512, 3), (4096, 3072, 1), (96, 2304, 2), (3072, 4096, 2)]:
        W, x = _case(oracle_mod, n, k, m, seed=7 * n + k)
        Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
        y = q4.q4_gemv(torch.from_numpy(W).cuda(), n, k, torch.from_numpy(x).cuda(), workspace=ws)
        ok, info = within_tol(y.cpu().numpy(), Y, S, TOL)
        assert ok, (n, k, m, info)
        torch.cuda.synchronize()
        assert int(ws.buf.count_nonzero().item()) == 0


@pytest.mark.parametrize("pdl", [False, True])
def test_gemv_prefetch_gives_q4_gemv_result(torch, q4, oracle_mod, pdl):
    """q4_gemv_prefetch is q4_gemv plus an L2 prefetch of another region: the
    result is q4_gemv's bit for bit (and within the oracle's bound), whether
    the region is another matrix, the call's own W or absent."""
    n, k = 4096, 3072
    W, x = _case(oracle_mod, n, k, 1, seed=77)
    W2, _ = _case(oracle_mod, 3072, 4096, 1, seed=78)
    Wd, xd, W2d = (torch.from_numpy(a).cuda() for a in (W, x, W2))
    flags = q4.FLAG_PDL if pdl else 0
    ref = q4.q4_gemv(Wd, n, k, xd, flags=flags).cpu().numpy()
    Y, S = oracle_mod.matmul(W, n, k, x)
    for region in (W2d, Wd, None):
        got = q4.q4_gemv_prefetch(Wd, n, k, xd, prefetch=region, flags=flags).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        ok, info = within_tol(got, Y, S, TOL)
        assert ok, info
