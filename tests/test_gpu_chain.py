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
    """Two 'layers' writing the same buffers, as a decoder step does: the chain's
    final output equals the sequential q4_gemv calls within the tolerance chain."""
    A, Ad = _mat(oracle_mod, torch, 2048, 1024, 7)
    B, Bd = _mat(oracle_mod, torch, 1024, 2048, 8)
    x0 = torch.from_numpy(synth.np_activations(1, 1024, seed=9)).cuda()
    h = torch.empty((1, 2048), device="cuda")
    out = torch.empty((1, 1024), device="cuda")
    links = [(Ad, 2048, 1024, x0, h), (Bd, 1024, 2048, h, out),
             (Ad, 2048, 1024, out, h), (Bd, 1024, 2048, h, out)]
    q4.q4_gemv_chain(links)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    # sequential reference through the oracle (fp32 between links)
    x = x0.cpu().numpy()
    for (W, n, k) in [(A, 2048, 1024), (B, 1024, 2048), (A, 2048, 1024), (B, 1024, 2048)]:
        y, _ = oracle_mod.matmul(W, n, k, x)
        x = y.astype(np.float32)
    rel = np.linalg.norm(got - y) / np.linalg.norm(y)
    assert rel < 1e-4, rel


def test_chain_decoder_step_matches_per_launch_step(torch, q4):
    """The 26-layer decode step as one chain vs 104 q4_gemv launches."""
    from bit_weight_quantized_03_b300.stacks import DecoderStack
    dec = DecoderStack(layers=3)
    x0 = synth.torch_activations(1, 3072, seed=synth.activation_seed(2000, 5))
    a = dec.step(x0).clone()
    b = dec.step(x0, chain=True).clone()
    torch.cuda.synchronize()
    rel = float((a - b).norm() / a.norm())
    assert rel < 1e-4, rel


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
