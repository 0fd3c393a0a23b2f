"""Parity at the benchmark's full sizes, in the launch configuration the benchmark
times (CUDA graphs, programmatic dependent launch, shared workspace).

Inputs come from the seeded generators in synth/ (device draws for the large
cases); expected values come only from the CPU oracle, computed from the same
generator output (regenerated fp32 weights copied to the host and quantized by
the oracle).  Where the oracle would take too long on the whole output, rows
are sampled; properties that hold at any size (exact power-of-two scaling,
run-to-run determinism, gather = decode of the same rows) cover the rest.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import bf16_round, same_float, within_tol

pytestmark = pytest.mark.gpu
GEMV_TOL, GEMM_TOL = 1e-4, 8e-3


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


def _graph_calls(torch, calls):
    """Run `calls` (callables taking a stream) once inside a captured CUDA graph."""
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for c in calls:
            c(s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c(s)
    g.replay()
    torch.cuda.synchronize()


def _oracle_rows(oracle_mod, torch, n, k, seed, rows):
    """Oracle-quantized blocks for `rows` of the seeded [n, k] weight matrix."""
    w = synth.torch_weights(n, k, seed=seed)[torch.as_tensor(rows, device="cuda")]
    blocks, rc, _ = oracle_mod.quantize(w.cpu().numpy())
    assert rc == 0
    return blocks


def _sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    r = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, count)]))
    return r


# --------------------------------------------------------------------- config 1

def test_config1_gemv_4096x3072_full(torch, q4, oracle_mod):
    n, k = 4096, 3072
    w = synth.np_weights(n, k, seed=synth.seed_for(1))
    W_ref, rc, _ = oracle_mod.quantize(w)
    assert rc == 0
    W_gpu = q4.q4_quantize(torch.from_numpy(w).cuda())
    assert np.array_equal(W_gpu.cpu().numpy(), W_ref)
    x = synth.np_activations(1, k, seed=synth.activation_seed(synth.seed_for(1)))
    Wd, xd = torch.from_numpy(W_ref).cuda(), torch.from_numpy(x).cuda()
    y = torch.empty((1, n), device="cuda")
    ws = q4.Workspace()
    _graph_calls(torch, [lambda s: q4.q4_gemv(Wd, n, k, xd, y=y, workspace=ws,
                                             flags=q4.FLAG_PDL, stream=s)])
    Y, S = oracle_mod.matmul(W_ref, n, k, x, nthreads=oracle_mod.cpu_count())
    ok, info = within_tol(y.cpu().numpy(), Y, S, GEMV_TOL)
    assert ok, info


# --------------------------------------------------------------------- config 2

@pytest.fixture(scope="module")
def decoder(torch):
    from bit_weight_quantized_03_b300.stacks import DecoderStack
    return DecoderStack()


MATS = [("wq", "qkv", 0, 4096, 3072, 0), ("wk", "qkv", 4096, 1024, 3072, 1),
        ("wv", "qkv", 5120, 1024, 3072, 2), ("wo", "wo", 0, 3072, 4096, 3),
        ("w1", "w13", 0, 9216, 3072, 4), ("w3", "w13", 9216, 9216, 3072, 5),
        ("w2", "w2", 0, 3072, 9216, 6)]


@pytest.mark.parametrize("layer", [0, 13, 25])
def test_config2_decoder_blocks_match_oracle(torch, oracle_mod, decoder, layer):
    for name, key, r0, n, k, idx in MATS:
        rows = _sample_rows(n, 24, seed=layer * 10 + idx)
        ref = _oracle_rows(oracle_mod, torch, n, k, synth.seed_for(2, layer, idx), rows)
        got = decoder.W[layer][key][torch.as_tensor(r0 + rows, device="cuda")].cpu().numpy()
        assert np.array_equal(got, ref), (layer, name)


def test_config2_all_104_gemvs_in_bench_launch_config(torch, q4, oracle_mod, decoder):
    """Every GEMV of a decode step, captured with PDL in one graph as the benchmark
    runs them, each on its own seeded input; sampled output rows vs the oracle."""
    outs, ins, calls = [], [], []
    for l in range(decoder.layers):
        for key, (n, k) in decoder.shapes.items():
            x = synth.torch_activations(1, k, seed=synth.activation_seed(synth.seed_for(2, l), 7))
            y = torch.empty((1, n), device="cuda")
            W = decoder.W[l][key]
            calls.append(lambda s, W=W, n=n, k=k, x=x, y=y: q4.q4_gemv(
                W, n, k, x, y=y, workspace=decoder.ws, flags=q4.FLAG_PDL, stream=s))
            outs.append((l, key, n, k, y))
            ins.append(x)
    _graph_calls(torch, calls)
    parts = {"qkv": [(4096, 0), (1024, 1), (1024, 2)], "wo": [(3072, 3)],
             "w13": [(9216, 4), (9216, 5)], "w2": [(3072, 6)]}
    for (l, key, n, k, y), x in zip(outs, ins):
        if l not in (0, 7, 25):
            continue
        r0 = 0
        for (pn, idx) in parts[key]:
            rows = _sample_rows(pn, 12, seed=l + idx)
            Wr = _oracle_rows(oracle_mod, torch, pn, k, synth.seed_for(2, l, idx), rows)
            Y, S = oracle_mod.matmul(Wr, len(rows), k, x.cpu().numpy())
            ok, info = within_tol(y.cpu().numpy()[:, r0 + rows], Y, S, GEMV_TOL)
            assert ok, (l, key, idx, info)
            r0 += pn


def test_config2_decode_step_exact_properties(torch, decoder):
    """Full 26-layer step: bit-identical on replay, and exactly scale-equivariant
    under a power of two (the chain of fp32 GEMVs is linear)."""
    x0 = synth.torch_activations(1, 3072, seed=synth.activation_seed(2000, 1))
    s = torch.cuda.Stream()
    g = decoder.capture([x0], s)
    g.replay()
    torch.cuda.synchronize()
    a = decoder.x.clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a, decoder.x)
    assert torch.isfinite(a).all()
    x0.mul_(2.0 ** -10)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(decoder.x, a * 2.0 ** -10)


def _oracle_mat(oracle_mod, torch, parts, l, rows=None):
    """Oracle-quantized blocks of a row-concatenated decoder matrix (rows: a
    subset of the concatenated rows, or all)."""
    k = parts[0][1]
    blocks, r0 = [], 0
    for (n, _, idx) in parts:
        sel = np.arange(n) if rows is None else rows[(rows >= r0) & (rows < r0 + n)] - r0
        if sel.size:
            blocks.append(_oracle_rows(oracle_mod, torch, n, k, synth.seed_for(2, l, idx), sel))
        r0 += n
    return np.concatenate(blocks), k


PARTS = {"qkv": [(4096, 3072, 0), (1024, 3072, 1), (1024, 3072, 2)], "wo": [(3072, 4096, 3)],
         "w13": [(9216, 3072, 4), (9216, 3072, 5)], "w2": [(3072, 9216, 6)]}


def test_config2_two_layer_step_each_product_vs_oracle(torch, q4, oracle_mod):
    """Two decoder layers through DecoderStack's per-launch step (PDL chain of
    q4_gemv), one layer at a time: every product element-wise against the
    oracle's fp64 product on the input that product read."""
    from bit_weight_quantized_03_b300.stacks import DecoderStack
    dec = DecoderStack(layers=2)
    th = oracle_mod.cpu_count()
    x = synth.torch_activations(1, 3072, seed=synth.activation_seed(2000, 2))
    for l in range(2):
        dec._layer(l, x, None)
        torch.cuda.synchronize()
        outs = {"qkv": dec.y_qkv.cpu().numpy(), "wo": dec.y_o.cpu().numpy(),
                "w13": dec.y_13.cpu().numpy(), "w2": dec.x.cpu().numpy()}
        ins = {"qkv": x.cpu().numpy(), "wo": outs["qkv"][:, :4096],
               "w13": outs["wo"], "w2": outs["w13"][:, :9216]}
        for key in ("qkv", "wo", "w13", "w2"):
            W, k = _oracle_mat(oracle_mod, torch, PARTS[key], l)
            n = W.shape[0]
            Y, S = oracle_mod.matmul(W, n, k, np.ascontiguousarray(ins[key]), nthreads=th)
            ok, info = within_tol(outs[key], Y, S, GEMV_TOL)
            assert ok, (l, key, info)
        x = dec.x.clone()


def _gated_bound(a, b, Sa, Sb, tol):
    """The product bounds tol*Sa, tol*Sb carried through g = a sigmoid(a) b,
    plus the fp32 rounding of the gate itself."""
    sig = 1.0 / (1.0 + np.exp(-a))
    g = a * sig * b
    return (tol * Sa * np.abs(b) * (sig + np.abs(a) * sig * (1 - sig)) +
            tol * Sb * np.abs(a * sig) + 1e-6 * np.abs(g) + 1e-30), g


def test_config2_fused_step_26_layers_sampled_vs_oracle(torch, q4, oracle_mod, decoder):
    """The full 26-layer decode step as one q4_chain on the repacked weights,
    with the gated FFN and both residual adds fused, every link writing its
    output: sampled rows of each of the 104 links element-wise against the
    oracle on the input that link read (weights from the oracle's own
    quantization of the seeded matrices).  The synthetic decoder has no norms
    (they are outside the Q4 path) and its gated FFN is quadratic in the scale
    of its input, so an N(0, 1) input overflows fp32 within a few layers; the
    input is scaled by 2^-24, which keeps all 26 layers finite (the slice
    scaling of the staged x is exact under powers of two)."""
    H, Q, F = 3072, 4096, 9216
    outs = []
    for l in range(decoder.layers):
        for n in (Q + 2048, H, F, H):
            outs.append(torch.full((n,), float("nan"), device="cuda"))
    x0 = synth.torch_activations(1, H, seed=synth.activation_seed(2000, 9)) * 2.0 ** -24
    decoder.fused_step(x0, outs=outs)
    torch.cuda.synchronize()
    got = [o.cpu().numpy().astype(np.float64) for o in outs]
    x_l = x0.cpu().numpy()[0]
    for l in range(decoder.layers):
        b = 4 * l
        y_qkv, h, g, x_next = got[b:b + 4]
        sel = lambda n, i: _sample_rows(n, 16, seed=1000 * l + i)  # noqa: E731
        # qkv = Wqkv x_l
        r = sel(Q + 2048, 0)
        W, k = _oracle_mat(oracle_mod, torch, PARTS["qkv"], l, r)
        Y, S = oracle_mod.matmul(W, len(r), k, x_l.astype(np.float32))
        ok, info = within_tol(y_qkv[r], Y[0], S[0], GEMV_TOL)
        assert ok, (l, "qkv", info)
        # h = x_l + Wo q
        r = sel(H, 1)
        W, k = _oracle_mat(oracle_mod, torch, PARTS["wo"], l, r)
        Y, S = oracle_mod.matmul(W, len(r), k, y_qkv[:Q].astype(np.float32))
        ok, info = within_tol(h[r], Y[0] + x_l[r], S[0] + np.abs(x_l[r]), GEMV_TOL)
        assert ok, (l, "wo + residual", info)
        # g = silu(W1 h) * (W3 h)
        r = sel(F, 2)
        W1, k = _oracle_mat(oracle_mod, torch, PARTS["w13"][:1], l, r)
        W3, _ = _oracle_mat(oracle_mod, torch, [(F, H, 5)], l, r)
        A, Sa = oracle_mod.matmul(W1, len(r), k, h.astype(np.float32))
        B, Sb = oracle_mod.matmul(W3, len(r), k, h.astype(np.float32))
        bound, gref = _gated_bound(A[0], B[0], Sa[0], Sb[0], GEMV_TOL)
        err = np.abs(g[r] - gref)
        assert np.all(err <= bound), (l, "gate", float(np.max(err / bound)))
        # x_{l+1} = h + W2 g
        r = sel(H, 3)
        W, k = _oracle_mat(oracle_mod, torch, PARTS["w2"], l, r)
        Y, S = oracle_mod.matmul(W, len(r), k, g.astype(np.float32))
        ok, info = within_tol(x_next[r], Y[0] + h[r], S[0] + np.abs(h[r]), GEMV_TOL)
        assert ok, (l, "w2 + residual", info)
        assert np.all(np.isfinite(x_next)), l
        x_l = x_next.astype(np.float32)


# --------------------------------------------------------------------- config 3

@pytest.fixture(scope="module")
def table(torch, q4):
    V, H, chunk = synth.VOCAB, 3072, 16384
    T = torch.empty((V, H // 32 * 18), dtype=torch.uint8, device="cuda")
    for c in range(V // chunk):
        w = synth.torch_weights(chunk, H, seed=synth.seed_for(3, 0, c))
        q4.q4_quantize(w, blocks=T[c * chunk:(c + 1) * chunk])
    torch.cuda.synchronize()
    return T


def _table_rows_ref(oracle_mod, torch, ids):
    chunk, H = 16384, 3072
    out = {}
    for c in sorted(set(int(i) // chunk for i in ids)):
        w = synth.torch_weights(chunk, H, seed=synth.seed_for(3, 0, c))
        sel = [int(i) for i in ids if int(i) // chunk == c]
        rows = w[torch.as_tensor([i - c * chunk for i in sel], device="cuda")].cpu().numpy()
        b, rc, _ = oracle_mod.quantize(rows)
        assert rc == 0
        for j, i in enumerate(sel):
            out[i] = b[j]
    return out


def test_config3_table_and_gather(torch, q4, oracle_mod, table):
    V, H = synth.VOCAB, 3072
    for B in (1, 64, 4096):
        ids = synth.torch_token_ids(B, V, seed=B)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty((B, H), device="cuda")
        _graph_calls(torch, [lambda s: q4.q4_embed_gather(table, V, H, ids, out=out, status=st,
                                                          stream=s)])
        assert int(st.item()) == 0
        ids_h = ids.cpu().numpy()
        pick = np.unique(np.concatenate([[0, B - 1], np.random.default_rng(B).integers(0, B, 24)]))
        ref_blocks = _table_rows_ref(oracle_mod, torch, ids_h[pick])
        for b in pick:
            blk = ref_blocks[int(ids_h[b])]
            assert np.array_equal(table[int(ids_h[b])].cpu().numpy(), blk)
            assert same_float(out[b].cpu().numpy(), oracle_mod.dequant_rows(blk, 1, H)[0])
        # every row: the gather equals the decode of the same rows
        rows = q4.q4_dequant_rows(table, 0, V, H)
        assert torch.equal(out, rows[ids.long()])
        del rows


def test_config3_head_gemv(torch, q4, oracle_mod, table):
    V, H = synth.VOCAB, 3072
    x = synth.torch_activations(1, H, seed=synth.activation_seed(3000))
    y = torch.empty((1, V), device="cuda")
    ws = q4.Workspace()
    _graph_calls(torch, [lambda s: q4.q4_gemv(table, V, H, x, y=y, workspace=ws,
                                             flags=q4.FLAG_PDL, stream=s)])
    pick = _sample_rows(V, 200, seed=3)
    ref = _table_rows_ref(oracle_mod, torch, pick)
    Wr = np.stack([ref[int(i)] for i in pick])
    Y, S = oracle_mod.matmul(Wr, len(pick), H, x.cpu().numpy())
    ok, info = within_tol(y.cpu().numpy()[:, pick], Y, S, GEMV_TOL)
    assert ok, info


# --------------------------------------------------------------------- config 4

@pytest.mark.parametrize("m", synth.ENCODER_FRAMES)
def test_config4_encoder_gemms(torch, q4, oracle_mod, m):
    X = synth.torch_activations(m, 1280, seed=synth.activation_seed(4000, m), dtype=torch.bfloat16)
    for idx, (name, n, k) in enumerate(synth.ENCODER_MATS):
        w = synth.torch_weights(n, k, seed=synth.seed_for(4, 0, idx))
        Wg = q4.q4_quantize(w)
        W_ref, rc, _ = oracle_mod.quantize(w.cpu().numpy())
        assert rc == 0 and np.array_equal(Wg.cpu().numpy(), W_ref)
        Xin = X if k == 1280 else synth.torch_activations(
            m, k, seed=synth.activation_seed(4100, m), dtype=torch.bfloat16)
        Y = torch.empty((m, n), device="cuda")
        _graph_calls(torch, [lambda s: q4.q4_gemm(Wg, n, k, Xin, Y=Y, flags=q4.FLAG_PDL,
                                                  stream=s)])
        toks = _sample_rows(m, 40, seed=m + idx)
        Yr, Sr = oracle_mod.matmul(W_ref, n, k, Xin.float().cpu().numpy()[toks],
                                   nthreads=oracle_mod.cpu_count())
        ok, info = within_tol(Y.cpu().numpy()[toks], Yr, Sr, GEMM_TOL)
        assert ok, (name, m, info)


# --------------------------------------------------------------------- config 5

@pytest.mark.parametrize("m", [1, 2, 4, 8, 16, 32, 64, 128])
def test_config5_crossover_shapes(torch, q4, oracle_mod, m):
    n, k = 4096, 3072
    w = synth.np_weights(n, k, seed=synth.seed_for(5))
    W, _, _ = oracle_mod.quantize(w)
    x = synth.np_activations(m, k, seed=synth.activation_seed(5000, m))
    Wd = torch.from_numpy(W).cuda()
    y = q4.q4_linear(Wd, n, k, torch.from_numpy(x).cuda()).cpu().numpy()
    gemv_path = m <= q4.q4_linear_crossover_m(n, k)
    Y, S = oracle_mod.matmul(W, n, k, x if gemv_path else bf16_round(x),
                             nthreads=oracle_mod.cpu_count())
    ok, info = within_tol(y, Y, S, GEMV_TOL if gemv_path else GEMM_TOL)
    assert ok, info
    if m <= q4.GEMV_MAX_M:
        yv = q4.q4_gemv(Wd, n, k, torch.from_numpy(x).cuda()).cpu().numpy()
        Y, S = oracle_mod.matmul(W, n, k, x, nthreads=oracle_mod.cpu_count())
        ok, info = within_tol(yv, Y, S, GEMV_TOL)
        assert ok, info
    xb = torch.from_numpy(x).to(torch.bfloat16)
    yg = q4.q4_gemm(Wd, n, k, xb.cuda()).cpu().numpy()
    Y, S = oracle_mod.matmul(W, n, k, xb.float().numpy(), nthreads=oracle_mod.cpu_count())
    ok, info = within_tol(yg, Y, S, GEMM_TOL)
    assert ok, info


# the measured crossover table of q4_linear (largest M sent to the fp32 GEMV)
CROSSOVER = {(4096, 3072): 4, (1024, 3072): 6, (3072, 4096): 4, (9216, 3072): 4,
             (3072, 9216): 4, (3840, 1280): 8, (1280, 1280): 6, (5120, 1280): 8,
             (1280, 5120): 6}


@pytest.mark.parametrize("shape", sorted(CROSSOVER))
def test_linear_at_each_shapes_crossover(torch, q4, oracle_mod, shape):
    """q4_linear at the measured crossover of every decoder and encoder shape
    and one row either side: the path it takes (fp32 GEMV up to the
    crossover, bf16 tensor-core GEMM past it) is checked element-wise against
    the oracle with that path's tolerance."""
    n, k = shape
    c = CROSSOVER[shape]
    assert q4.q4_linear_crossover_m(n, k) == c
    W, rc, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=synth.seed_for(5, 2, n + k)))
    assert rc == 0
    Wd = torch.from_numpy(W).cuda()
    for m in (c - 1, c, c + 1):
        x = synth.np_activations(m, k, seed=synth.activation_seed(5200 + n + k, m))
        y = q4.q4_linear(Wd, n, k, torch.from_numpy(x).cuda()).cpu().numpy()
        gemv = m <= c
        Y, S = oracle_mod.matmul(W, n, k, x if gemv else bf16_round(x),
                                 nthreads=oracle_mod.cpu_count())
        ok, info = within_tol(y, Y, S, GEMV_TOL if gemv else GEMM_TOL)
        assert ok, (shape, m, info)
