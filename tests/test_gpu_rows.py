"""GPU parity of the row kernels through the C ABI: quantize, dequant (fp32 and
bf16) and the embedding-row gather are bit-exact against the CPU oracle."""
import numpy as np
import pytest

import synth
from conftest import parse_values, read_golden
from gpu_helpers import bf16_round, same_float

pytestmark = pytest.mark.gpu

SHAPES = [(1, 32), (3, 288), (17, 96), (257, 3072), (64, 9216), (5, 4096)]


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


@pytest.mark.parametrize("n,k", SHAPES)
def test_quantize_bit_exact(torch, q4, oracle_mod, n, k):
    w = synth.np_weights(n, k, seed=n * 7 + k)
    ref, rc, _ = oracle_mod.quantize(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = q4.q4_quantize(torch.from_numpy(w).cuda(), status=st)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    assert np.array_equal(got.cpu().numpy(), ref)


def test_quantize_hand_derived_blocks(torch, q4, oracle_mod):
    rows = read_golden("quantize_blocks.txt")
    w = np.stack([parse_values(r[1]) for r in rows]).astype(np.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = q4.q4_quantize(torch.from_numpy(w).cuda(), status=st).cpu().numpy()
    for i, r in enumerate(rows):
        assert got[i].tobytes().hex() == r[3], r[0]
    # at least one of the golden blocks is non-finite
    assert int(st.item()) == q4.ERR_NONFINITE


def test_quantize_distributions(torch, q4, oracle_mod):
    rng = np.random.default_rng(99)
    w = np.concatenate([
        rng.standard_normal((8, 512)).astype(np.float32) * np.float32(1e-6),
        rng.standard_normal((8, 512)).astype(np.float32) * np.float32(3e3),
        rng.uniform(-1, 1, (8, 512)).astype(np.float32),
        (rng.standard_normal((8, 512)) * 1e-7).astype(np.float32)])
    w[3, 100] = -w[3, 101]
    w[5, 0:32] = 0.0
    w[6, 32:64] = -0.0
    ref, _, _ = oracle_mod.quantize(w)
    got = q4.q4_quantize(torch.from_numpy(w).cuda()).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("n,k", SHAPES)
def test_dequant_rows_fp32_bf16(torch, q4, oracle_mod, n, k):
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=3 + n))
    ref = oracle_mod.dequant_rows(W, n, k)
    Wd = torch.from_numpy(W).cuda()
    got = q4.q4_dequant_rows(Wd, 0, n, k).cpu().numpy()
    assert same_float(got, ref)
    gotb = q4.q4_dequant_rows(Wd, 0, n, k, out_dtype=torch.bfloat16).float().cpu().numpy()
    assert same_float(gotb, bf16_round(ref))
    if n > 2:  # a row window starting inside the matrix
        r0 = n // 2
        sub = q4.q4_dequant_rows(Wd, r0, n - r0, k).cpu().numpy()
        assert same_float(sub, ref[r0:])


def test_dequant_hand_built_blocks(torch, q4):
    rows = read_golden("decode_blocks.txt")
    W = np.frombuffer(b"".join(bytes.fromhex(r[1]) for r in rows), np.uint8).copy()
    W16 = np.zeros(((W.size + 15) // 16) * 16, np.uint8)
    W16[:W.size] = W
    got = q4.q4_dequant_rows(torch.from_numpy(W16).cuda(), 0, len(rows), 32).cpu().numpy()
    for i, r in enumerate(rows):
        assert same_float(got[i], parse_values(r[2])), r[0]


@pytest.mark.parametrize("vocab,k,b", [(1, 32, 1), (50, 288, 7), (1000, 3072, 64), (4096, 3072, 513)])
def test_gather_bit_exact(torch, q4, oracle_mod, vocab, k, b):
    T, _, _ = oracle_mod.quantize(synth.np_weights(vocab, k, seed=vocab + k))
    ids = synth.np_token_ids(b, vocab, seed=b)
    ref, rc = oracle_mod.embed_gather(T, vocab, k, ids)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = q4.q4_embed_gather(torch.from_numpy(T).cuda(), vocab, k, torch.from_numpy(ids).cuda(),
                             status=st).cpu().numpy()
    assert rc == 0 and int(st.item()) == 0
    assert same_float(got, ref)


def test_gather_out_of_range_ids(torch, q4, oracle_mod):
    vocab, k = 100, 256
    T, _, _ = oracle_mod.quantize(synth.np_weights(vocab, k, seed=1))
    ids = np.array([0, 99, 100, -1, 5, 2 ** 31 - 1, 50], np.int32)
    ref, rc = oracle_mod.embed_gather(T, vocab, k, ids)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = q4.q4_embed_gather(torch.from_numpy(T).cuda(), vocab, k, torch.from_numpy(ids).cuda(),
                             status=st).cpu().numpy()
    torch.cuda.synchronize()
    assert rc == q4.ERR_ID_OUT_OF_RANGE
    assert int(st.item()) == q4.ERR_ID_OUT_OF_RANGE
    assert same_float(got, ref)
