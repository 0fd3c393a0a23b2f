"""The repacked layout (q4_repack), the repacked batch-1 GEMV (q4_gemv_r) and the
fused decode-step chain (q4_chain), called through the C ABI and compared with
the CPU oracle on the same seeded inputs:

* q4_repack is bit-exact against the oracle's own statement of the layout;
* q4_gemv_r meets |y - y_ref| <= 1e-4 * sum_j |w^ x| element by element on
  shapes that span many tiles, ragged 16-row groups, groups split between
  SMs and k up to the kernel's 12288; unit vectors give the decoded columns
  exactly, all-8 codes give zeros, power-of-two scaling is exact, and results
  do not change from run to run;
* q4_chain runs a small decoder (the gated FFN unit in the epilogue of the
  w1/w3 product, two residual adds per layer) and an argmax head in one launch;
  each link is checked against the oracle applied to the input it read, built
  from the chain's own earlier outputs, within 1e-4 * (sum |w^ x| + |residual|);
  the gated outputs against the oracle's fp64 gate of its own w1/w3 products,
  within that bound carried through the gate's derivatives; the argmax is a
  valid maximum of the oracle's logits within the tolerance and the
  lowest-index maximum of the chain's own logits;
* the workspace carries over from call to call (and between chains of
  different shapes), and a call whose bounded wait runs out reports
  Q4_ERR_TIMEOUT.
"""
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


def _quant(oracle_mod, n, k, seed):
    W, rc, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=seed))
    assert rc == 0
    return W


def _repacked(torch, q4, W, n, k):
    return q4.q4_repack(torch.from_numpy(W).cuda(), n, k)


# ------------------------------------------------------------------ q4_repack

@pytest.mark.parametrize("n,k", [(1, 256), (16, 256), (17, 512), (37, 768), (100, 3072),
                                 (1000, 9216), (33, 12288)])
def test_repack_bit_exact(torch, q4, oracle_mod, n, k):
    rng = np.random.default_rng(n * 7 + k)
    W = rng.integers(0, 256, size=(n, k // 32 * 18), dtype=np.uint8)
    R = q4.q4_repack(torch.from_numpy(W).cuda(), n, k).cpu().numpy()
    assert R.size == q4.q4_repack_bytes(n, k) == oracle_mod.repack_bytes(n, k)
    assert np.array_equal(R, oracle_mod.repack(W, n, k))


# ------------------------------------------------------------------ q4_gemv_r

GEMV_SHAPES = [(1, 256), (16, 256), (17, 512), (33, 768), (4096, 3072), (1000, 3072),
               (3072, 4096), (6144, 3072), (3072, 9216), (257, 9216), (100, 12288),
               (18432, 3072), (130, 1280), (2, 2560)]


@pytest.mark.parametrize("n,k", GEMV_SHAPES)
def test_gemv_r_matches_oracle(torch, q4, oracle_mod, n, k):
    W = _quant(oracle_mod, n, k, seed=n + 3 * k)
    x = synth.np_activations(1, k, seed=n + k + 1)
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    R = _repacked(torch, q4, W, n, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = q4.q4_gemv_r(R, n, k, torch.from_numpy(x).cuda(), status=st,
                     workspace=q4.Workspace()).cpu().numpy()
    assert int(st.item()) == 0
    ok, info = within_tol(y, Y, S, TOL)
    assert ok, info


def test_gemv_r_unit_vectors_give_columns(torch, q4, oracle_mod):
    n, k = 77, 512
    W = _quant(oracle_mod, n, k, seed=8)
    cols = oracle_mod.dequant_rows(W, n, k).T  # [k, n]
    R = _repacked(torch, q4, W, n, k)
    ws = q4.Workspace()
    for j in list(range(0, k, 37)) + [k - 1]:
        x = np.zeros((1, k), np.float32)
        x[0, j] = 1.0
        y = q4.q4_gemv_r(R, n, k, torch.from_numpy(x).cuda(), workspace=ws).cpu().numpy()
        assert np.array_equal(y[0], cols[j]), j  # exact (+0 and -0 compare equal)


def test_gemv_r_all_eight_codes_give_zero(torch, q4):
    n, k = 70, 768
    W = np.zeros((n, k // 32 * 18), np.uint8)
    blk = W.reshape(n, k // 32, 18)
    blk[:, :, 0:2] = np.frombuffer(np.float16(-2.75).tobytes(), np.uint8)
    blk[:, :, 2:] = 0x88
    x = synth.np_activations(1, k, seed=3)
    R = _repacked(torch, q4, W, n, k)
    y = q4.q4_gemv_r(R, n, k, torch.from_numpy(x).cuda(), workspace=q4.Workspace())
    assert bool(torch.all(y == 0).item())


def test_gemv_r_power_of_two_scaling_and_determinism(torch, q4, oracle_mod):
    n, k = 4096, 3072
    W = _quant(oracle_mod, n, k, seed=21)
    x = synth.np_activations(1, k, seed=22)
    R = _repacked(torch, q4, W, n, k)
    ws = q4.Workspace()
    xd = torch.from_numpy(x).cuda()
    ys = [q4.q4_gemv_r(R, n, k, xd, workspace=ws).cpu().numpy() for _ in range(3)]
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint32), ys[0].view(np.uint32))
    y2 = q4.q4_gemv_r(R, n, k, xd * (2.0 ** -6), workspace=ws).cpu().numpy()
    assert np.array_equal(y2, ys[0] * np.float32(2.0 ** -6))


def test_gemv_r_timeout_then_recovers(torch, q4, oracle_mod):
    n, k = 4096, 3072
    W = _quant(oracle_mod, n, k, seed=31)
    x = synth.np_activations(1, k, seed=32)
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
    R = _repacked(torch, q4, W, n, k)
    ws = q4.Workspace()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xd = torch.from_numpy(x).cuda()
    q4.q4_gemv_r(R, n, k, xd, workspace=ws, status=st, flags=q4.FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert int(st.item()) == q4.ERR_TIMEOUT
    ws.reset()  # a device error: the workspace is zero-filled again
    st.zero_()
    y = q4.q4_gemv_r(R, n, k, xd, workspace=ws, status=st).cpu().numpy()
    assert int(st.item()) == 0
    ok, info = within_tol(y, Y, S, TOL)
    assert ok, info


# ------------------------------------------------------------------ q4_chain

H, QD, KVD, F, V = 256, 512, 128, 768, 1000


class _Decoder:
    """Two layers of the decoder's linears at small sizes, plus a head."""

    def __init__(self, torch, q4, oracle_mod, layers=2, seed=0):
        self.layers = []
        for l in range(layers):
            s = 5000 + 10 * l + seed
            mats = {"qkv": (QD + 2 * KVD, H, s), "wo": (H, QD, s + 1), "w2": (H, F, s + 3)}
            lay = {}
            for name, (n, k, sd) in mats.items():
                W = _quant(oracle_mod, n, k, sd)
                lay[name] = (W, n, k, _repacked(torch, q4, W, n, k))
            # w1 (gate) and w3 (up), interleaved 8 rows at a time for the gate epilogue
            W1, W3 = _quant(oracle_mod, F, H, s + 2), _quant(oracle_mod, F, H, s + 4)
            W13 = q4.interleave_gate_rows(torch.from_numpy(W1), torch.from_numpy(W3)).numpy()
            lay["w13"] = (W13, 2 * F, H, _repacked(torch, q4, W13, 2 * F, H), W1, W3)
            self.layers.append(lay)
        Wh = _quant(oracle_mod, V, H, 5900 + seed)
        self.head = (Wh, V, H, _repacked(torch, q4, Wh, V, H))

    def links(self, torch, q4, x_in, outs, argmax, head_y=True):
        L = []
        for l, lay in enumerate(self.layers):
            b = 4 * l
            x_l = x_in if l == 0 else q4.LinkOut(b - 1)
            W, n, k, R = lay["qkv"]
            L.append(q4.Link(R, n, k, x_l, y=outs[b]))
            W, n, k, R = lay["wo"]
            L.append(q4.Link(R, n, k, q4.LinkOut(b, 0), y=outs[b + 1], residual=x_l,
                             ops=q4.OP_RESIDUAL))
            W, n, k, R = lay["w13"][:4]
            L.append(q4.Link(R, n, k, q4.LinkOut(b + 1), y=outs[b + 2], ops=q4.OP_SWIGLU))
            W, n, k, R = lay["w2"]
            L.append(q4.Link(R, n, k, q4.LinkOut(b + 2), residual=q4.LinkOut(b + 1),
                             y=outs[b + 3], ops=q4.OP_RESIDUAL))
        W, n, k, R = self.head
        L.append(q4.Link(R, n, k, q4.LinkOut(len(L) - 1), y=outs[-1] if head_y else None,
                         argmax=argmax, ops=q4.OP_ARGMAX))
        return L

    def out_buffers(self, torch):
        outs = []
        for lay in self.layers:
            for name in ("qkv", "wo", "w13", "w2"):
                n = lay[name][1] // (2 if name == "w13" else 1)  # the gate halves w1/w3
                outs.append(torch.full((n,), float("nan"), device="cuda"))
        outs.append(torch.full((V,), float("nan"), device="cuda"))
        return outs


def _check(got, Y, S, R=None, what=""):
    bound = TOL * (S + (np.abs(R) if R is not None else 0.0))
    err = np.abs(got.astype(np.float64) - Y)
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, (what, [(int(i), float(got[i]), float(Y[i]), float(bound[i]))
                                  for i in bad[:5, 0]])


def _check_chain(oracle_mod, dec, x_in, outs_np, am):
    th = oracle_mod.cpu_count()
    x_l = x_in.astype(np.float32)
    for l, lay in enumerate(dec.layers):
        b = 4 * l
        y_qkv, h, y13, x_next = outs_np[b:b + 4]
        W, n, k, _ = lay["qkv"]
        Y, S = oracle_mod.matmul(W, n, k, x_l, nthreads=th)
        _check(y_qkv, Y[0], S[0], what=f"layer {l} qkv")
        W, n, k, _ = lay["wo"]
        Y, S = oracle_mod.matmul(W, n, k, y_qkv[:QD], nthreads=th)
        _check(h, Y[0] + x_l.astype(np.float64), S[0], x_l.astype(np.float64),
               what=f"layer {l} wo + residual")
        W1, W3 = lay["w13"][4], lay["w13"][5]
        A1, S1 = oracle_mod.matmul(W1, F, H, h, nthreads=th)
        A3, S3 = oracle_mod.matmul(W3, F, H, h, nthreads=th)
        a, b3 = A1[0], A3[0]
        g_ref = oracle_mod.swiglu(a, b3)
        sig = 1.0 / (1.0 + np.exp(-a))
        # the products' bound carried through the gate: |dg/da| <= |b| (sig + |a| sig (1-sig)),
        # |dg/db| = |a sig|; plus the fp32 rounding of the gate itself
        bound = (TOL * S1[0] * np.abs(b3) * (sig + np.abs(a) * sig * (1 - sig)) +
                 TOL * S3[0] * np.abs(a * sig) + 1e-6 * np.abs(g_ref) + 1e-30)
        err = np.abs(y13.astype(np.float64) - g_ref)
        assert np.all(err <= bound), (l, float(np.max(err / bound)))
        W, n, k, _ = lay["w2"]
        Y, S = oracle_mod.matmul(W, n, k, y13, nthreads=th)
        _check(x_next, Y[0] + h.astype(np.float64), S[0], h.astype(np.float64),
               what=f"layer {l} w2 + residual")
        x_l = x_next
    W, n, k, _ = dec.head
    Y, S = oracle_mod.matmul(W, n, k, x_l, nthreads=th)
    logits = outs_np[-1]
    _check(logits, Y[0], S[0], what="head")
    i = int(am[0])
    # a valid maximum of the oracle's logits within the tolerance ...
    tol = TOL * S[0]
    assert Y[0][i] + tol[i] >= np.max(Y[0] - tol)
    # ... and exactly the lowest-index maximum of the chain's own logits
    assert i == int(np.flatnonzero(logits == logits.max())[0])
    assert am[1] == logits[i].view(np.int32)


def test_chain_decoder_links_match_oracle(torch, q4, oracle_mod):
    dec = _Decoder(torch, q4, oracle_mod)
    x_in = synth.np_activations(1, H, seed=77)[0]
    outs = dec.out_buffers(torch)
    am = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = q4.Workspace()
    links = dec.links(torch, q4, torch.from_numpy(x_in).cuda(), outs, am)
    q4.q4_chain(links, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_chain(oracle_mod, dec, x_in, [o.cpu().numpy() for o in outs], am.cpu().numpy())


def test_chain_repeats_bitwise_and_shares_workspace(torch, q4, oracle_mod):
    """Consecutive launches on one workspace (alternating slot sets), with a
    chain of another shape in between, give bitwise the same results."""
    dec = _Decoder(torch, q4, oracle_mod)
    other = _Decoder(torch, q4, oracle_mod, layers=1, seed=3)
    x_in = torch.from_numpy(synth.np_activations(1, H, seed=78)[0]).cuda()
    ws = q4.Workspace()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    runs = []
    for r in range(5):
        if r == 2:
            o2 = other.out_buffers(torch)
            am2 = torch.zeros(2, dtype=torch.int32, device="cuda")
            q4.q4_chain(other.links(torch, q4, x_in, o2, am2), workspace=ws, status=st)
        outs = dec.out_buffers(torch)
        am = torch.zeros(2, dtype=torch.int32, device="cuda")
        q4.q4_chain(dec.links(torch, q4, x_in, outs, am), workspace=ws, status=st)
        torch.cuda.synchronize()
        runs.append(([o.cpu().numpy() for o in outs], am.cpu().numpy()))
    assert int(st.item()) == 0
    for outs_np, am_np in runs[1:]:
        for a, b in zip(outs_np, runs[0][0]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(am_np, runs[0][1])
    _check_chain(oracle_mod, dec, x_in.cpu().numpy(), runs[0][0], runs[0][1])


def test_chain_argmax_without_logits(torch, q4, oracle_mod):
    """The head's argmax with y not written equals the one with y written."""
    dec = _Decoder(torch, q4, oracle_mod, layers=1, seed=5)
    x_in = torch.from_numpy(synth.np_activations(1, H, seed=79)[0]).cuda()
    ws = q4.Workspace()
    outs = dec.out_buffers(torch)
    am1 = torch.zeros(2, dtype=torch.int32, device="cuda")
    q4.q4_chain(dec.links(torch, q4, x_in, outs, am1), workspace=ws)
    outs2 = dec.out_buffers(torch)
    am2 = torch.zeros(2, dtype=torch.int32, device="cuda")
    q4.q4_chain(dec.links(torch, q4, x_in, outs2, am2, head_y=False), workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(am1.cpu().numpy(), am2.cpu().numpy())
    assert bool(torch.isnan(outs2[-1]).all().item())  # the logits were never written


def test_chain_argmax_ties_and_nan(torch, q4):
    """Rows with equal values: the lowest index wins; NaN rows never win.
    Weights: every code 8 (zeros) except chosen rows, x = ones."""
    n, k = 600, 256
    W = np.zeros((n, k // 32 * 18), np.uint8)
    blk = W.reshape(n, k // 32, 18)
    blk[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    blk[:, :, 2:] = 0x88
    blk[[101, 377, 599], 0, 2] = 0x8F  # element 0 code 15 -> +7 on these rows
    blk[50, :, 0:2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)  # 0 * inf = NaN
    Rw = q4.q4_repack(torch.from_numpy(W).cuda(), n, k)
    x = torch.ones(k, device="cuda")
    am = torch.zeros(2, dtype=torch.int32, device="cuda")
    y = torch.empty(n, device="cuda")
    q4.q4_chain([q4.Link(Rw, n, k, x, y=y, argmax=am, ops=q4.OP_ARGMAX)], workspace=q4.Workspace())
    torch.cuda.synchronize()
    assert torch.isnan(y[50]).item() and float(y[101].item()) == 7.0
    assert int(am[0].item()) == 101
    assert am.cpu().numpy()[1] == np.float32(7.0).view(np.int32)


def test_chain_timeout_reports_and_recovers(torch, q4, oracle_mod):
    dec = _Decoder(torch, q4, oracle_mod, layers=1, seed=7)
    x_np = synth.np_activations(1, H, seed=80)[0]
    x_in = torch.from_numpy(x_np).cuda()
    ws = q4.Workspace()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = dec.out_buffers(torch)
    am = torch.zeros(2, dtype=torch.int32, device="cuda")
    q4.q4_chain(dec.links(torch, q4, x_in, outs, am), workspace=ws, status=st,
                flags=q4.FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert int(st.item()) == q4.ERR_TIMEOUT
    ws.reset()
    st.zero_()
    outs = dec.out_buffers(torch)
    q4.q4_chain(dec.links(torch, q4, x_in, outs, am), workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_chain(oracle_mod, dec, x_np, [o.cpu().numpy() for o in outs], am.cpu().numpy())


def test_gemv_r_pdl_dependent_calls_in_a_graph(torch, q4, oracle_mod):
    """q4_gemv_r with Q4_FLAG_PDL (the half-size CTA shape, launched as a
    programmatic dependent launch), captured in a CUDA graph as a chain of
    dependent calls: y1 = A x, y2 = B y1, y3 = A' y2 ... each call's weights
    are read before the previous call ends, its x only after.  Every output
    element-wise against the oracle on the input that call read."""
    shapes = [(512, 768), (256, 512), (1024, 256), (768, 1024)]
    mats, Rs = [], []
    for i, (n, k) in enumerate(shapes):
        W = _quant(oracle_mod, n, k, 900 + i)
        mats.append(W)
        Rs.append(_repacked(torch, q4, W, n, k))
    x0 = torch.from_numpy(synth.np_activations(1, 768, seed=901)).cuda()
    ys = [torch.full((1, n), float("nan"), device="cuda") for n, _ in shapes]
    ws = q4.Workspace()
    s = torch.cuda.Stream()

    def run():
        src = x0
        for (n, k), R, y in zip(shapes, Rs, ys):
            q4.q4_gemv_r(R, n, k, src, y=y, workspace=ws, flags=q4.FLAG_PDL, stream=s)
            src = y
    with torch.cuda.stream(s):
        run()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run()
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
    s.synchronize()
    inp = x0.cpu().numpy()
    for (n, k), W, y in zip(shapes, mats, ys):
        got = y.cpu().numpy()
        Y, S = oracle_mod.matmul(W, n, k, inp)
        _check(got[0], Y[0], S[0], what=f"{n}x{k}")
        inp = got
