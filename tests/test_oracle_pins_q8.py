"""Pins of the oracle's Q4 x Q8 integer path (READING: the usual companion of
GGUF Q4_0, GeekNews es.news.hada.io/topic?id=26595, "Arquitectura"; the
pages give no detail, the reading is stated in oracle/q4_oracle.h):

* the per-32 int8 quantization of x on blocks whose codes are known exactly
  (a power-of-two scale, halves rounded away from zero, zero and non-finite
  blocks), and by brute force (no other code is nearer, in exact rationals);
* the product's factorization d_w d_x sum (q_w - 8) q_x against the plain sum
  of dequantized weight times dequantized activation, in exact rationals;
* its error against the unquantized fp64 product (at most half an x step per
  element, weighted by |w|), and exact scaling under powers of two.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def o():
    import oracle
    return oracle


def test_q8_exact_codes_on_power_of_two_scale(o):
    # amax = 127 * 2^-3 -> d = 2^-3 exactly, so x = c * 2^-3 has code c
    c = np.array([127, -127, 0, 1, -1, 5, -64, 100] + list(range(-12, 12)), np.float32)
    x = c * np.float32(0.125)
    q, d = o.quantize_q8(x)
    assert d[0] == np.float32(0.125)
    assert np.array_equal(q.astype(np.int64), c.astype(np.int64))
    # the largest magnitude negative: d from |x|, codes keep their sign
    c2 = np.array([-127, 10, -3, 0] + [1] * 28, np.float32)
    q, d = o.quantize_q8(c2 * np.float32(0.25))
    assert d[0] == np.float32(0.25)
    assert np.array_equal(q.astype(np.int64), c2.astype(np.int64))


def test_q8_rounds_halves_away_from_zero(o):
    # amax = 127 -> d = 1: x / d is x itself
    x = np.zeros(32, np.float32)
    x[:9] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -0.49]
    q, d = o.quantize_q8(x)
    assert d[0] == 1.0
    assert list(q[:9]) == [127, 3, -3, 1, -1, 2, -2, 127, 0]


def test_q8_zero_and_nonfinite_blocks(o):
    x = np.zeros(96, np.float32)
    x[40] = np.nan
    x[64:] = 1.0
    x[70] = np.inf
    q, d = o.quantize_q8(x)
    assert d[0] == 0 and not np.signbit(d[0]) and np.all(q[:32] == 0)
    assert np.isnan(d[1]) and np.all(q[32:64] == 0)
    assert np.isnan(d[2]) and np.all(q[64:] == 0)


def test_q8_codes_are_nearest_by_brute_force(o):
    rng = np.random.default_rng(3)
    for trial in range(20):
        x = (rng.standard_normal(32) * 10.0 ** rng.integers(-3, 4)).astype(np.float32)
        q, d = o.quantize_q8(x)
        D = Fraction(float(d[0]))
        for j in range(32):
            X = Fraction(float(x[j]))
            t = X / D
            frac = abs(t - int(t))
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10 ** 5):
                continue  # a near-tie: the fp32 quotient decides
            best = min(range(-127, 128), key=lambda cc: (abs(X - cc * D), -abs(cc)))
            assert int(q[j]) == best, (trial, j)


def test_q8_product_equals_dequantized_sum_exactly(o):
    """sum_b d_w d_x sum_j (q_w - 8) q_x == sum_j w^_j * (q_x_j d_x), exactly."""
    n, k = 3, 96
    W, rc, _ = o.quantize(synth.np_weights(n, k, seed=51))
    assert rc == 0
    x = synth.np_activations(1, k, seed=52)[0]
    q, d = o.quantize_q8(x)
    Y, S = o.matmul_q8(W, n, k, x)
    for r in range(n):
        wrow = o.dequant_rows(W, n, k)[r]
        exact = sum(Fraction(float(wrow[j])) * q[j] * Fraction(float(d[j // 32]))
                    for j in range(k))
        assert abs(Fraction(Y[0, r]) - exact) <= Fraction(S[0, r]) * Fraction(1, 2 ** 50)


def test_q8_error_against_unquantized_product(o):
    n, k = 17, 256
    W, _, _ = o.quantize(synth.np_weights(n, k, seed=53))
    x = synth.np_activations(1, k, seed=54)[0]
    _, d = o.quantize_q8(x)
    Yq, _ = o.matmul_q8(W, n, k, x)
    Y, S = o.matmul(W, n, k, x)
    w = o.dequant_rows(W, n, k).astype(np.float64)
    bound = (np.abs(w) * np.repeat(d.astype(np.float64) / 2, 32)[None, :]).sum(axis=1)
    assert np.all(np.abs(Yq[0] - Y[0]) <= bound + 1e-12 * S[0])


def test_q8_power_of_two_scaling_is_exact(o):
    n, k = 5, 128
    W, _, _ = o.quantize(synth.np_weights(n, k, seed=55))
    x = synth.np_activations(1, k, seed=56)[0]
    q1, d1 = o.quantize_q8(x)
    q2, d2 = o.quantize_q8(x * np.float32(32.0))
    assert np.array_equal(q1, q2) and np.array_equal(d2, d1 * np.float32(32.0))
    Y1, _ = o.matmul_q8(W, n, k, x)
    Y2, _ = o.matmul_q8(W, n, k, x * np.float32(32.0))
    assert np.array_equal(Y2, Y1 * 32.0)
