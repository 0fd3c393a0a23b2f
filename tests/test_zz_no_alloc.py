"""q4_gemv_noalloc through the C ABI: the GEMV entry point for callers that
cannot allocate device memory (a host embedding this library in a fixed memory
pool with cudaMalloc forbidden, a real-time loop that must not allocate once
streaming has started, a plugin handed only its input and output buffers).

Its split-K scratch is one fixed array inside the library, shared by every
call, so the test makes several calls in a row -- different shapes, so that a
call that started from the previous call's leftovers would show -- and checks
each element-wise against the CPU oracle's fp64 product and against the
existing q4_gemv entry point (its own zero-filled workspace), within the GEMV
tolerance |y - y_ref| <= 1e-4 * sum_j |w^ x|; then a call whose bounded wait
runs out is followed by a normal call that must be correct with no reset.
This file is collected last on purpose.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import within_tol

pytestmark = pytest.mark.gpu
TOL = 1e-4

# (n, k, m): config-1 shape, a ragged split-K shape with m = 3, then the first again
CALLS = [(4096, 3072, 1), (1000, 3072, 3), (4096, 3072, 1)]


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
    w = synth.np_weights(n, k, seed=seed)
    x = synth.np_activations(m, k, seed=seed + 50)
    W, rc, _ = oracle_mod.quantize(w)
    assert rc == 0
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    return W, x, Y, S


def test_noalloc_matches_oracle_and_q4_gemv_on_calls_in_a_row(torch, q4, oracle_mod):
    for i, (n, k, m) in enumerate(CALLS):
        W, x, Y, S = _case(oracle_mod, n, k, m, seed=900 + i)
        Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
        y_ref = q4.q4_gemv(Wd, n, k, xd, workspace=q4.Workspace()).cpu().numpy()
        # output and status word allocated before the call: the call itself allocates nothing
        y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q4.q4_gemv_noalloc(Wd, n, k, xd, y=y, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got = y.cpu().numpy()
        ok, info = within_tol(got, Y, S, TOL)  # element-wise against the fp64 oracle
        assert ok, (i, n, k, m, info)
        err = np.abs(got.astype(np.float64) - y_ref.astype(np.float64))
        assert np.all(err <= TOL * S), (i, n, k, m, float(np.max(err / np.maximum(S, 1e-30))))


def test_noalloc_call_after_a_timed_out_call(torch, q4, oracle_mod):
    """A call whose bounded wait runs out (test flag) may leave partial sums in
    the shared scratch; the next call clears what it uses, so it is correct
    without any reset by the caller."""
    n, k, m = 4096, 3072, 1
    W, x, Y, S = _case(oracle_mod, n, k, m, seed=990)
    Wd, xd = torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda()
    y = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q4.q4_gemv_noalloc(Wd, n, k, xd, y=y, status=st, flags=q4.FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert int(st.item()) == q4.ERR_TIMEOUT
    st.zero_()
    y.fill_(float("nan"))
    q4.q4_gemv_noalloc(Wd, n, k, xd, y=y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ok, info = within_tol(y.cpu().numpy(), Y, S, TOL)
    assert ok, info


def test_noalloc_rejects_sizes_beyond_its_scratch(q4):
    """A shape whose split-K scratch exceeds the fixed array is refused on the
    host with Q4_ERR_UNSUPPORTED_SHAPE before anything is launched (the
    addresses below are never dereferenced)."""
    L = q4.lib()
    n, k, m = 1 << 20, 3072, 16
    assert L.q4_gemv_workspace_bytes(n, k, m) > q4.GEMV_NOALLOC_SCRATCH_BYTES
    fake = 0x7F0000000000
    st = L.q4_gemv_noalloc(fake, n, k, fake, m, k, fake, n, None, 0, None)
    assert st == q4.ERR_UNSUPPORTED_SHAPE
