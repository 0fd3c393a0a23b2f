"""q4_gemv_chain through the C ABI: a chain of dependent batch-1 products in one
persistent launch.  Each link's output is checked against the fp64 oracle applied
to the exact input that link read (the previous link's output as the chain
produced it), |y - y_ref| <= 1e-4 * sum_j |w^ x|; plus run-to-run determinism,
the workspace counter returning to zero, buffer reuse between links, and the
host-side argument checks."""
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


def _mat(oracle_mod, torch, n, k, seed):
    W, rc, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=seed))
    assert rc == 0
    return W, torch.from_numpy(W).cuda()


def test_chain_links_match_oracle(torch, q4, oracle_mod):
    # (n, k, x source): "ext" = its own input, "prev" = previous y (from an offset)
    spec = [(4096, 3072, "ext", 0), (3072, 4096, "prev", 0), (6144, 3072, "prev", 0),
            (256, 512, "prev", 1024), (9216, 256, "prev", 0), (3072, 9216, "prev", 0),
            (100, 3072, "prev", 0), (40, 768, "ext", 0)]
    mats, ys, links, ins = [], [], [], []
    for i, (n, k, src, off) in enumerate(spec):
        Wn, Wd = _mat(oracle_mod, torch, n, k, 100 + i)
        y = torch.full((1, n), float("nan"), device="cuda")
        if src == "ext":
            x = torch.from_numpy(synth.np_activations(1, k, seed=200 + i)).cuda()
        else:
            x = ys[-1][:, off:off + k]
        mats.append((Wn, n, k))
        ys.append(y)
        ins.append(x)
        links.append((Wd, n, k, x, y))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = q4.Workspace()
    q4.q4_gemv_chain(links, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    th = oracle_mod.cpu_count()
    for i, ((Wn, n, k), x, y) in enumerate(zip(mats, ins, ys)):
        Y, S = oracle_mod.matmul(Wn, n, k, x.cpu().numpy(), nthreads=th)
        ok, info = within_tol(y.cpu().numpy(), Y, S, TOL)
        assert ok, (i, info)
    nb = q4.q4_gemv_chain_workspace_bytes(links)
    assert int(ws.buf[:256].count_nonzero().item()) == 0  # barrier counter back at zero
    # deterministic: a second run gives the same bits
    first = [y.clone() for y in ys]
    q4.q4_gemv_chain(links, workspace=ws, status=st)
    torch.cuda.synchronize()
    for a, b in zip(first, ys):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert nb > 256


def test_chain_reuses_buffers_like_sequential_calls(torch, q4, oracle_mod):
    """Two 'layers' writing the same buffers, as a decoder step does: links 3
    and 4 overwrite what links 1 and 2 read and wrote.  The chain is run once
    whole and once cut after link 2 (the outputs of links 1-2 then stay in
    place), and each link's output is checked element-wise against the
    oracle's product on the input it read."""
    A, Ad = _mat(oracle_mod, torch, 2048, 1024, 7)
    B, Bd = _mat(oracle_mod, torch, 1024, 2048, 8)
    x0 = torch.from_numpy(synth.np_activations(1, 1024, seed=9)).cuda()
    h = torch.empty((1, 2048), device="cuda")
    out = torch.empty((1, 1024), device="cuda")
    first = [(Ad, 2048, 1024, x0, h), (Bd, 1024, 2048, h, out)]
    q4.q4_gemv_chain(first)
    torch.cuda.synchronize()
    h1, out1 = h.cpu().numpy(), out.cpu().numpy()
    q4.q4_gemv_chain(first + [(Ad, 2048, 1024, out, h), (Bd, 1024, 2048, h, out)])
    torch.cuda.synchronize()
    h2, out2 = h.cpu().numpy(), out.cpu().numpy()
    th = oracle_mod.cpu_count()
    for (W, n, k), x, y in [((A, 2048, 1024), x0.cpu().numpy(), h1), ((B, 1024, 2048), h1, out1),
                            ((A, 2048, 1024), out1, h2), ((B, 1024, 2048), h2, out2)]:
        Y, S = oracle_mod.matmul(W, n, k, x, nthreads=th)
        ok, info = within_tol(y, Y, S, TOL)
        assert ok, (n, k, info)


def test_chain_decoder_step_each_link_vs_oracle(torch, q4, oracle_mod):
    """Three decoder layers (qkv, wo, w1|w3, w2 at full size) as one
    q4_gemv_chain, each link writing its own buffer: every link element-wise
    against the oracle's product on the input that link read."""
    shapes = [(6144, 3072), (3072, 4096), (18432, 3072), (3072, 9216)]
    mats, links, outs = [], [], []
    x = torch.from_numpy(synth.np_activations(1, 3072, seed=11)).cuda()
    first = x
    for l in range(3):
        for i, (n, k) in enumerate(shapes):
            W, Wd = _mat(oracle_mod, torch, n, k, 100 + 4 * l + i)
            y = torch.empty((1, n), device="cuda")
            src = x if i == 0 else outs[-1][:, :k]
            links.append((Wd, n, k, src, y))
            mats.append((W, n, k))
            outs.append(y)
        x = outs[-1]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q4.q4_gemv_chain(links, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    th = oracle_mod.cpu_count()
    inp = first.cpu().numpy()
    for (W, n, k), y in zip(mats, outs):
        got = y.cpu().numpy()
        Y, S = oracle_mod.matmul(W, n, k, np.ascontiguousarray(inp[:, :k]), nthreads=th)
        ok, info = within_tol(got, Y, S, TOL)
        assert ok, (n, k, info)
        inp = got


def test_chain_host_checks(torch, q4):
    """Arguments the host rejects before anything is launched."""
    L = q4.lib()
    W0 = torch.zeros((512, 512 // 32 * 18), dtype=torch.uint8, device="cuda")
    W1 = torch.zeros((64, 256 // 32 * 18), dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 512), device="cuda")
    y0 = torch.zeros((1, 512), device="cuda")
    y1 = torch.zeros((1, 64), device="cuda")
    arr = q4._chain_array
    # k not a multiple of 256
    assert L.q4_gemv_chain(arr([(W0, 512, 288, x, y0)]), 1, None, 0, None, 0, None) == \
        q4.ERR_UNSUPPORTED_SHAPE
    # link 1 reads link 0's y from an offset that is not a multiple of 4 floats
    bad = [(W0, 512, 512, x, y0), (W1, 64, 256, y0[:, 2:258], y1)]
    assert L.q4_gemv_chain(arr(bad), 2, None, 0, None, 0, None) in (q4.ERR_INVALID_ARG,
                                                                    q4.ERR_MISALIGNED)
    # no links / too many
    assert L.q4_gemv_chain(arr([(W0, 512, 512, x, y0)]), 0, None, 0, None, 0, None) == \
        q4.ERR_INVALID_ARG
    # a valid chain without its workspace
    good = [(W0, 512, 512, x, y0), (W1, 64, 256, y0[:, 4:260], y1)]
    assert L.q4_gemv_chain(arr(good), 2, None, 0, None, 0, None) == q4.ERR_WORKSPACE
