"""Pins for the oracle's decoder-glue and layout functions, each tied to
something other than the oracle itself:

* the repacked tile layout against byte offsets derived by hand from its
  definition (tests/golden/repack_offsets.txt), and the exact round trip;
* the SiLU-gated unit (the gated FFN activation reading) against the known
  value sigmoid(1) = 1/(1 + 1/e), the identity silu(x) - silu(-x) = x, its
  limits and its exact linearity in the up input;
* argmax against hand-built cases (ties, NaN, all-NaN) and a brute-force
  search on random data with planted ties;
* the fp64-input product against the fp32-input one on fp32 values and
  against exact rational arithmetic on inputs that are not fp32 values.
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
import synth


# ------------------------------------------------------------------ repacked layout

def _marked_matrix(oracle_mod, n, k, seed):
    """Random Q4_0 blocks whose bytes are all distinct enough to locate."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(n, k // 32 * 18), dtype=np.uint8)


def _nibble(W, nb, r, kb, e):
    byte = W[r, kb * 18 + 2 + (e % 16)]
    return int(byte & 0xF) if e < 16 else int(byte >> 4)


def test_repack_hand_derived_offsets(oracle_mod):
    n, k = 20, 512
    W = _marked_matrix(oracle_mod, n, k, seed=3)
    R = oracle_mod.repack(W, n, k)
    assert R.size == oracle_mod.repack_bytes(n, k) == 9216
    rows = read_golden("repack_offsets.txt")
    assert len(rows) == 7
    for row, blk, el, so, co, half in rows:
        r, kb, e, so, co = int(row), int(blk), int(el), int(so), int(co)
        assert R[so] == W[r, kb * 18] and R[so + 1] == W[r, kb * 18 + 1], (r, kb)
        got = int(R[co] & 0xF) if half == "low" else int(R[co] >> 4)
        assert got == _nibble(W, k // 32, r, kb, e), (r, kb, e)
    # padding row 31, block 0 (hand-derived in the golden file's comments)
    assert R[4834] == 0 and R[4835] == 0
    assert np.all(R[5312:5320] == 0x88)


@pytest.mark.parametrize("n,k", [(1, 256), (16, 256), (37, 768), (64, 3072)])
def test_repack_round_trip(oracle_mod, n, k):
    W = _marked_matrix(oracle_mod, n, k, seed=n + k)
    R = oracle_mod.repack(W, n, k)
    assert np.array_equal(oracle_mod.unrepack(R, n, k), W)


def test_repack_padding_rows_decode_to_zero(oracle_mod):
    """Every byte of the padding rows is d = +0 / code 8, and the repacked size
    counts whole 16-row groups."""
    n, k = 17, 256
    W = _marked_matrix(oracle_mod, n, k, seed=9)
    R = oracle_mod.repack(W, n, k)
    assert R.size == 2 * 2304
    W32 = oracle_mod.unrepack(R, 32, k)  # read the padding rows back as rows 17..31
    assert np.all(W32[17:, 0::18] == 0) and np.all(W32[17:, 1::18] == 0)
    codes = np.concatenate([W32[17:, 2 + 18 * b:18 + 18 * b] for b in range(8)], axis=1)
    assert np.all(codes == 0x88)


def test_repack_rejects_bad_shapes(oracle_mod):
    assert oracle_mod.repack_bytes(4, 288) == 0
    assert oracle_mod.repack_bytes(0, 256) == 0


# ------------------------------------------------------------------ SiLU-gated unit

def test_swiglu_known_values(oracle_mod):
    sig1 = 0.7310585786300049  # 1 / (1 + 1/e)
    got = oracle_mod.swiglu([0.0, 1.0, -1.0, 1.0], [5.0, 1.0, 1.0, 3.0])
    assert got[0] == 0.0
    assert got[1] == pytest.approx(sig1, rel=1e-15)
    assert got[2] == pytest.approx(-(1.0 - sig1), rel=1e-15)
    assert got[3] == pytest.approx(3 * sig1, rel=1e-15)


def test_swiglu_odd_part_identity(oracle_mod):
    """sigmoid(x) + sigmoid(-x) = 1, so silu(x) - silu(-x) = x."""
    x = synth.np_activations(1, 4096, seed=21).ravel().astype(np.float64) * 4
    ones = np.ones_like(x)
    d = oracle_mod.swiglu(x, ones) - oracle_mod.swiglu(-x, ones)
    assert np.allclose(d, x, rtol=1e-14, atol=1e-15)


def test_swiglu_limits_and_linearity(oracle_mod):
    got = oracle_mod.swiglu([50.0, -50.0], [1.0, 1.0])
    assert got[0] == 50.0
    assert got[1] < 0 and abs(got[1]) < 1e-18
    a = synth.np_activations(1, 512, seed=22).ravel().astype(np.float64)
    b = synth.np_activations(1, 512, seed=23).ravel().astype(np.float64)
    assert np.array_equal(oracle_mod.swiglu(a, 2 * b), 2 * oracle_mod.swiglu(a, b))
    assert np.array_equal(oracle_mod.swiglu(a, -b), -oracle_mod.swiglu(a, b))


# ------------------------------------------------------------------ argmax

def test_argmax_hand_built(oracle_mod):
    assert oracle_mod.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle_mod.argmax([np.nan, 1.0, 0.0]) == 1
    assert oracle_mod.argmax([0.0, np.nan, 2.0, np.nan]) == 2
    assert oracle_mod.argmax([np.nan, np.nan]) == -1
    assert oracle_mod.argmax([-np.inf, -np.inf]) == 0
    assert oracle_mod.argmax([-1.0, -0.5, -2.0]) == 1
    assert oracle_mod.argmax([]) == -1


def test_argmax_brute_force(oracle_mod):
    rng = np.random.default_rng(31)
    for trial in range(20):
        y = rng.integers(-5, 6, size=200).astype(np.float64)  # many ties
        if trial % 3 == 0:
            y[rng.integers(0, 200, size=7)] = np.nan
        best = max(v for v in y if not np.isnan(v))
        first = next(i for i, v in enumerate(y) if v == best)
        assert oracle_mod.argmax(y) == first


# ------------------------------------------------------------------ fp64-input product

def test_matmul_f64_equals_fp32_path_on_fp32_inputs(oracle_mod):
    n, k = 37, 512
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=41))
    x = synth.np_activations(2, k, seed=42)
    Y32, S32 = oracle_mod.matmul(W, n, k, x)
    Y64, S64 = oracle_mod.matmul_f64(W, n, k, x.astype(np.float64))
    assert np.array_equal(Y32, Y64) and np.array_equal(S32, S64)


def test_matmul_f64_exact_on_tiny_shapes(oracle_mod):
    n, k = 3, 64
    W, _, _ = oracle_mod.quantize(synth.np_weights(n, k, seed=43))
    w = oracle_mod.dequant_rows(W, n, k).astype(np.float64)
    x = np.array([(-1) ** i / (3 + i) for i in range(k)], np.float64)  # not fp32 values
    Y, S = oracle_mod.matmul_f64(W, n, k, x)
    for r in range(n):
        exact = sum(Fraction(float(w[r, j])) * Fraction(float(x[j])) for j in range(k))
        sabs = sum(abs(Fraction(float(w[r, j])) * Fraction(float(x[j]))) for j in range(k))
        assert abs(Fraction(Y[0, r]) - exact) <= Fraction(k) * Fraction(2) ** -52 * sabs
        assert S[0, r] == pytest.approx(float(sabs), rel=1e-13)
