"""Pins for the oracle's product with x quantized to int8 (activation
quantization, "oxinfer" crate page, How it works: per-matmul activation
quantization ahead of int8 dot products).

The reading: per 32 elements of x, s = max|x| / 127 (fp32), codes
q = round(x / s) (fp32 division, ties away from zero) in -127..127, and the
product sum_k w * s * q.  The pins hold it to facts outside its own code:
blocks that are exact multiples of a power-of-two scale reduce to the pinned
fp32-x oracle, every code is within half a step of x, half-way values go away
from zero, zero blocks vanish, power-of-two scaling and sign flips carry
through exactly, and the result stays within the quantization error bound of
the exact product.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


def exact_multiples(rng, M, K, e):
    """x = 2^-e * q with integer q in -127..127 and |q| = 127 somewhere in
    every block of 32: the rule then recovers q and s = 2^-e exactly."""
    q = rng.integers(-127, 128, (M, K))
    q[:, ::32] = np.where(rng.random((M, K // 32)) < 0.5, 127, -127)
    return (q * 2.0 ** -e).astype(np.float32), q


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_exact_multiples_reduce_to_the_fp32_product(fmt):
    rng = np.random.default_rng((100, fmt))
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 37, 4 * be, 3
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(101, fmt))
    x, q = exact_multiples(rng, M, K, 9)
    xq, sc = oracle.quantize_x_int8(x)
    assert np.array_equal(xq, q) and np.all(sc == 2.0 ** -9)
    y8, b8 = oracle.qmatmul_x_int8(fmt, W, x, N, K)
    y, b = oracle.qmatmul(fmt, W, x, N, K)
    assert np.array_equal(y8, y) and np.array_equal(b8, b)


def test_codes_within_half_a_step():
    rng = np.random.default_rng(102)
    x = (rng.standard_normal((4, 2048)) * np.exp(rng.uniform(-8, 8, (4, 1)))).astype(np.float32)
    x[0, 100] = 1e4  # an outlier channel
    xq, sc = oracle.quantize_x_int8(x)
    s = np.repeat(sc.astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - s * xq)
    assert np.all(err <= 0.5 * s * (1 + 2.0 ** -20))
    assert np.all(np.abs(xq) <= 127)
    # the largest element of every block gets the extreme code
    blk = np.abs(x).reshape(4, -1, 32)
    amax_pos = blk.argmax(axis=2)
    codes = np.abs(xq.reshape(4, -1, 32))
    assert np.all(np.take_along_axis(codes, amax_pos[..., None], axis=2) == 127)


def test_ties_go_away_from_zero():
    """s = 1 exactly (max |x| = 127); x = k + 0.5 -> k + 1, -(k + 0.5) -> -(k + 1)."""
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0
    x[0, 1:9] = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5]
    xq, sc = oracle.quantize_x_int8(x)
    assert sc[0, 0] == 1.0
    assert list(xq[0, :9]) == [127, 1, 2, 3, 4, -1, -2, -3, -4]


def test_zero_block_and_scaling_and_sign():
    rng = np.random.default_rng(103)
    fmt, N, K = syn.Q8_0, 20, 128
    W, x = syn.make_problem(fmt, N, K, 2, seed=(104,))
    x[:, 32:64] = 0.0
    xq, sc = oracle.quantize_x_int8(x)
    assert np.all(xq[:, 32:64] == 0) and np.all(sc[:, 1] == 0)
    y, b = oracle.qmatmul_x_int8(fmt, W, x, N, K)
    for e in (-5, 7):
        ys, bs = oracle.qmatmul_x_int8(fmt, W, x * np.float32(2.0 ** e), N, K)
        assert np.array_equal(ys, y * 2.0 ** e) and np.array_equal(bs, b * 2.0 ** e)
    yn, bn = oracle.qmatmul_x_int8(fmt, W, -x, N, K)
    assert np.array_equal(yn, -y) and np.array_equal(bn, b)
    # a zero block contributes nothing: zeroing it in x changes nothing
    x2 = x.copy()
    x2[:, 32:64] = 0.0
    y2, _ = oracle.qmatmul_x_int8(fmt, W, x2, N, K)
    assert np.array_equal(y2, y)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_within_the_quantization_bound_of_the_exact_product(fmt):
    """|y_int8x - y| <= sum_k |w_k| * s_b(k) / 2 (each code within half a step)."""
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 50, 8 * be, 2
    W, x = syn.make_problem(fmt, N, K, M, seed=(105, fmt))
    y8, _ = oracle.qmatmul_x_int8(fmt, W, x, N, K)
    y, _ = oracle.qmatmul(fmt, W, x, N, K)
    w = np.abs(oracle.dequant(fmt, W, N, K))
    _, sc = oracle.quantize_x_int8(x)
    s = np.repeat(sc.astype(np.float64), 32, axis=1)  # [M][K]
    lim = 0.5 * (s @ w.T) * (1 + 1e-6)
    assert np.all(np.abs(y8 - y) <= lim)
    # and it is a real approximation: far outside the exact product's tolerance
    _, b = oracle.qmatmul(fmt, W, x, N, K)
    assert np.mean(np.abs(y8 - y) > 1e-4 * b + 1e-6) > 0.5
