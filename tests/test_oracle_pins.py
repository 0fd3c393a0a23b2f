"""Pins for the CPU oracle: each check ties it to something other than itself.

* binary16 conversions against numpy's own float16 (an independent library);
* block decode against hand-derived literal values (tests/golden/decode_blocks.txt);
* quantize against hand-derived blocks (tests/golden/quantize_blocks.txt), the
  round-trip error bound, idempotence, and brute-force optimality of every code;
* the fp64 product against exact rational arithmetic (fractions) on tiny shapes,
  against numpy's float64 matmul, closed-form special cases and exact scaling.
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import parse_values, read_golden
import synth


def _same_float(a: np.ndarray, b: np.ndarray) -> bool:
    """Bit-for-bit equality, except that any NaN matches any NaN."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    nan = np.isnan(a) & np.isnan(b)
    eq = a.view(np.uint32) == b.view(np.uint32)
    return bool(np.all(nan | eq))


# ------------------------------------------------------------------ binary16

def test_half_to_float_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle_mod.half_to_float(int(b)) for b in bits], np.float32)
    assert _same_float(got, ref)


def test_float_to_half_rne_against_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(20000).astype(np.float32) * np.float32(s)
            for s in (1e-8, 1e-6, 1e-4, 1.0, 1e2, 1e4, 7e4)]
    # every halfway point between consecutive binary16 values, and one fp32 ulp on
    # each side of it: the cases where rounding direction and ties-to-even matter
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    vals += [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    vals += [np.array([0.0, -0.0, 65504, 65519.996, 65520, 65536, 1e30, np.inf, -np.inf,
                       2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26], np.float32)]
    x = np.concatenate(vals)
    x = np.concatenate([x, -x])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref), x[got != ref][:10]
    assert oracle_mod.float_to_half(float("nan")) & 0x7C00 == 0x7C00


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("row", read_golden("decode_blocks.txt"), ids=lambda r: r[0])
def test_decode_hand_built(oracle_mod, row):
    name, hexbytes, values = row
    expect = parse_values(values)
    got = oracle_mod.decode_block(bytes.fromhex(hexbytes))
    assert expect.size == 32
    assert _same_float(got, expect), (name, got, expect)


def test_decode_rows_match_block_decode(oracle_mod):
    rng = np.random.default_rng(11)
    n, k = 5, 96
    W = rng.integers(0, 256, size=(n, k // 32 * 18), dtype=np.uint8)
    # keep scales finite so the comparison below is on numbers
    for b in range(k // 32):
        W[:, b * 18 + 1] &= 0x7B
    rows = oracle_mod.dequant_rows(W, n, k)
    for r in range(n):
        for b in range(k // 32):
            blk = W[r, b * 18:(b + 1) * 18].tobytes()
            assert _same_float(rows[r, b * 32:(b + 1) * 32], oracle_mod.decode_block(blk))


# ------------------------------------------------------------------ quantize

@pytest.mark.parametrize("row", read_golden("quantize_blocks.txt"), ids=lambda r: r[0])
def test_quantize_hand_derived(oracle_mod, row):
    name, values, status, hexbytes = row
    x = parse_values(values)
    assert x.size == 32
    blk, rc = oracle_mod.quantize_block(x)
    assert rc == int(status), name
    assert blk.hex() == hexbytes, (name, blk.hex(), hexbytes)


def _blocks_of(W, n, k):
    return W.reshape(n, k // 32, 18)


def _quantize_cases():
    rng = np.random.default_rng(2024)
    cases = [synth.np_weights(64, 256, seed=1)]
    cases.append(rng.standard_normal((16, 256)).astype(np.float32) * np.float32(1e3))
    cases.append(rng.uniform(-1, 1, (16, 256)).astype(np.float32))
    heavy = rng.standard_normal((16, 256)).astype(np.float32)
    heavy[:, ::7] *= 50
    cases.append(heavy)
    sym = rng.standard_normal((8, 256)).astype(np.float32)
    sym[:, 1] = -sym[:, 0]  # +a and -a in one block: the clamped case
    cases.append(sym)
    return cases


@pytest.mark.parametrize("ci", range(5))
def test_quantize_roundtrip_bound(oracle_mod, ci):
    """|w - w^| <= |d|/2 (plus fp32 rounding slack) for every unclamped element;
    <= |d| for an element clamped to code 0 or 15 (the +a/-a case)."""
    w = _quantize_cases()[ci]
    n, k = w.shape
    W, rc, bad = oracle_mod.quantize(w)
    assert rc == 0 and bad == 0
    deq = oracle_mod.dequant_rows(W, n, k).astype(np.float64)
    blocks = _blocks_of(W, n, k)
    d = blocks[:, :, 0:2].copy().view(np.float16).astype(np.float64)[..., 0]
    dd = np.repeat(d, 32, axis=1)
    err = np.abs(w.astype(np.float64) - deq)
    t = w.astype(np.float64) / np.where(dd == 0, 1, dd)
    clamped = (t + 8.5 >= 16) | (t + 8.5 < 0)
    slack = 2.0 ** -18
    assert np.all(err[~clamped] <= np.abs(dd[~clamped]) * (0.5 + slack))
    assert np.all(err[clamped] <= np.abs(dd[clamped]) * (1.0 + 2.0 ** -9))


@pytest.mark.parametrize("ci", range(5))
def test_quantize_codes_are_optimal(oracle_mod, ci):
    """Brute force: no other code gives a smaller |x - (q-8)*dd| (near-ties allowed
    within the fp32 rounding of x/dd + 8.5)."""
    w = _quantize_cases()[ci][:4]
    n, k = w.shape
    W, _, _ = oracle_mod.quantize(w)
    blocks = _blocks_of(W, n, k)
    for r in range(n):
        for b in range(k // 32):
            blk = blocks[r, b]
            dd = float(blk[0:2].copy().view(np.float16)[0])
            qs = blk[2:18]
            codes = np.concatenate([qs & 0xF, qs >> 4]).astype(np.int64)
            x = w[r, b * 32:(b + 1) * 32].astype(np.float64)
            cand = (np.arange(16)[None, :] - 8) * dd
            errs = np.abs(x[:, None] - cand)
            best = errs.min(axis=1)
            chosen = errs[np.arange(32), codes]
            assert np.all(chosen <= best + abs(dd) * 2.0 ** -18)


def test_quantize_idempotent(oracle_mod):
    """quantize(dequant(quantize(w))) == quantize(w) bit for bit (normal scales)."""
    for ci, w in enumerate(_quantize_cases()):
        n, k = w.shape
        W1, _, _ = oracle_mod.quantize(w)
        W2, rc, _ = oracle_mod.quantize(oracle_mod.dequant_rows(W1, n, k))
        assert rc == 0
        assert np.array_equal(W1, W2), ci


def test_quantize_nonfinite_rows_flagged(oracle_mod):
    w = synth.np_weights(3, 64, seed=5)
    w[1, 40] = np.nan
    W, rc, bad = oracle_mod.quantize(w)
    assert rc == 4 and bad == 1
    blk = _blocks_of(W, 3, 64)[1, 1]
    assert blk.tobytes() == bytes(2) + bytes([0x88] * 16)


# ------------------------------------------------------------------ fp64 product

def _np_decode(W, n, k):
    """Independent restatement of the block decode with numpy, used only to feed
    the exact rational sums below."""
    blocks = _blocks_of(W, n, k)
    d = blocks[:, :, 0:2].copy().view(np.float16).astype(np.float32)  # [n, nb, 1]
    qs = blocks[:, :, 2:18].astype(np.int32)
    q = np.concatenate([qs & 0xF, qs >> 4], axis=2) - 8
    return (q.astype(np.float32) * d).reshape(n, k)


@pytest.mark.parametrize("n,k,m", [(1, 32, 1), (2, 64, 3), (3, 256, 1), (17, 64, 3), (17, 256, 3)])
def test_matmul_brute_force_exact(oracle_mod, n, k, m):
    w = synth.np_weights(n, k, seed=100 + n * k)
    x = synth.np_activations(m, k, seed=200 + m)
    W, _, _ = oracle_mod.quantize(w)
    Y, S = oracle_mod.matmul(W, n, k, x)
    deq = _np_decode(W, n, k)
    assert np.array_equal(deq, oracle_mod.dequant_rows(W, n, k))
    for mm in range(m):
        for i in range(n):
            exact = sum(Fraction(float(deq[i, j])) * Fraction(float(x[mm, j])) for j in range(k))
            sabs = sum(abs(Fraction(float(deq[i, j])) * Fraction(float(x[mm, j]))) for j in range(k))
            assert abs(Fraction(Y[mm, i]) - exact) <= Fraction(k) * Fraction(2) ** -53 * sabs
            assert abs(Fraction(S[mm, i]) - sabs) <= Fraction(k) * Fraction(2) ** -53 * sabs


def test_matmul_against_numpy_float64(oracle_mod):
    n, k, m = 300, 1024, 4
    w = synth.np_weights(n, k, seed=3)
    x = synth.np_activations(m, k, seed=4)
    W, _, _ = oracle_mod.quantize(w)
    Y, S = oracle_mod.matmul(W, n, k, x, nthreads=3)
    deq = _np_decode(W, n, k).astype(np.float64)
    ref = x.astype(np.float64) @ deq.T
    sref = np.abs(x.astype(np.float64)[:, None, :] * deq[None, :, :]).sum(-1)
    assert np.all(np.abs(Y - ref) <= 1e-12 * sref)
    assert np.allclose(S, sref, rtol=1e-12, atol=0)


def test_matmul_threads_do_not_change_results(oracle_mod):
    n, k, m = 257, 512, 2
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=8))
    x = synth.np_activations(m, k, seed=9)
    Y1, S1 = oracle_mod.matmul(W, n, k, x, nthreads=1)
    Y4, S4 = oracle_mod.matmul(W, n, k, x, nthreads=4)
    assert np.array_equal(Y1, Y4) and np.array_equal(S1, S4)


def test_matmul_unit_vectors_give_columns(oracle_mod):
    n, k = 9, 96
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=12))
    eye = np.eye(k, dtype=np.float32)
    Y, _ = oracle_mod.matmul(W, n, k, eye)
    assert np.array_equal(Y.T.astype(np.float32), _np_decode(W, n, k))


def test_matmul_zero_codes_give_zero(oracle_mod):
    n, k = 4, 64
    W = np.zeros((n, k // 32 * 18), np.uint8)
    blocks = _blocks_of(W, n, k)
    blocks[:, :, 0:2] = np.frombuffer(np.float16(3.5).tobytes(), np.uint8)
    blocks[:, :, 2:] = 0x88
    Y, S = oracle_mod.matmul(W, n, k, synth.np_activations(2, k, seed=1))
    assert np.all(Y == 0) and np.all(S == 0)


def test_matmul_scales_exactly_with_d_and_x(oracle_mod):
    """Multiplying every d by 2^3 (binary16 exponent +3) or x by 2^-5 scales Y and S
    exactly: the decoded weights and every product scale by the same power of two."""
    n, k, m = 6, 128, 2
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=13))
    x = synth.np_activations(m, k, seed=14)
    Y, S = oracle_mod.matmul(W, n, k, x)
    W8 = W.copy()
    blocks = _blocks_of(W8, n, k)
    dbits = blocks[:, :, 0:2].copy().view(np.uint16)
    assert np.all(((dbits >> 10) & 0x1F) < 28)  # stays normal and finite
    blocks[:, :, 0:2] = (dbits + (3 << 10)).view(np.uint8)
    Y8, S8 = oracle_mod.matmul(W8, n, k, x)
    assert np.array_equal(Y8, Y * 8) and np.array_equal(S8, S * 8)
    Yx, Sx = oracle_mod.matmul(W, n, k, x * np.float32(2.0 ** -5))
    assert np.array_equal(Yx, Y * 2.0 ** -5) and np.array_equal(Sx, S * 2.0 ** -5)


def test_matmul_linear_in_x(oracle_mod):
    n, k = 10, 256
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=15))
    x1 = synth.np_activations(1, k, seed=16)
    x2 = synth.np_activations(1, k, seed=17)
    Y1, S1 = oracle_mod.matmul(W, n, k, x1)
    Y2, S2 = oracle_mod.matmul(W, n, k, x2)
    Y12, _ = oracle_mod.matmul(W, n, k, x1 + x2)
    assert np.all(np.abs(Y12 - (Y1 + Y2)) <= 1e-6 * (S1 + S2))


# ------------------------------------------------------------------ gather

def test_gather_rows_and_out_of_range(oracle_mod):
    vocab, k = 50, 96
    T, _, _ = oracle_mod.quantize(synth.np_weights(vocab, k, seed=21))
    ids = np.array([0, 49, 7, 7, 3], np.int32)
    out, rc = oracle_mod.embed_gather(T, vocab, k, ids)
    assert rc == 0
    rows = oracle_mod.dequant_rows(T, vocab, k)
    assert _same_float(out, rows[ids])
    out, rc = oracle_mod.embed_gather(T, vocab, k, np.array([1, 50, -1, 2], np.int32))
    assert rc == 5
    assert _same_float(out[0], rows[1]) and _same_float(out[3], rows[2])
    assert np.all(out[1:3].view(np.uint32) == 0)  # +0.0


def test_invalid_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.quantize(np.zeros((2, 48), np.float32))
    with pytest.raises(ValueError):
        oracle_mod.matmul(np.zeros(18, np.uint8), 1, 32, np.zeros((1, 31), np.float32))
