"""Pins for the oracle's float -> block quantizers (CPU).

The pages quantize weights at load time ("oxinfer" crate page, How it works:
quant.rs; "wgpu-llm" README, INT8 mode) without a rounding rule; the oracle
takes the reading written at the top of its quantizer section.  These tests
hold it to things other than itself: numpy's correctly rounded double -> half
conversion, hand-worked blocks, and a brute-force search over every code for
the nearest one.
"""
import numpy as np
import pytest

import oracle

Q4_0, Q8_0, I8_B64 = 0, 1, 2


def half_bits(v):
    with np.errstate(over="ignore"):  # past 65504 numpy gives Inf; the tests check that case
        return int(np.array([v], np.float64).astype(np.float16).view(np.uint16)[0])


def test_fp16_rounding_matches_numpy():
    """Nearest binary16 (ties to even), normal and subnormal, both signs,
    including every half-way point between neighbouring binary16 values."""
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(20000) * np.exp2(rng.integers(-30, 16, 20000)))
    h = np.arange(0, 0x7bff, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2  # exact in double
    vals += list(mids[::7]) + list(-mids[::11]) + [0.0, -0.0, 65504.0, 65519.99, 2.0 ** -25]
    for v in vals:
        ref = half_bits(v)
        got = oracle.double_to_fp16(v)
        if ref & 0x7fff == 0x7c00:  # numpy overflowed to Inf: the oracle refuses
            assert got == -1, v
        else:
            assert got == ref, v
    assert oracle.double_to_fp16(65520.0) == -1
    assert oracle.double_to_fp16(float("nan")) == -1


def test_q8_hand_worked_block():
    # max |w| = 63.5 -> d = 0.5 exactly; 0.25 / 0.5 = 0.5 rounds away from zero
    w = np.zeros(32, np.float32)
    w[:6] = [63.5, -63.5, 0.5, 0.25, -0.25, 0.74]
    blk = oracle.quantize(Q8_0, w, 1, 32)
    assert blk[:2].view(np.uint16)[0] == 0x3800  # 0.5
    assert list(blk[2:8].view(np.int8)) == [127, -127, 1, 1, -1, 1]
    assert (blk[8:] == 0).all()


def test_q4_0_hand_worked_blocks():
    # negative extreme m = -8: d = 1, q = round(w) + 8
    w = np.zeros(32, np.float32)
    w[:6] = [-8.0, 7.0, 3.5, -3.5, 0.49, 7.6]
    blk = oracle.quantize(Q4_0, w, 1, 32)
    assert blk[:2].view(np.uint16)[0] == 0x3C00  # 1.0
    q = [(blk[2 + j] & 15) if j < 16 else (blk[2 + j - 16] >> 4) for j in range(32)]
    assert q[:6] == [0, 15, 12, 4, 8, 15]  # 3.5 -> 4, -3.5 -> -4, 7.6 -> 8 clamps to 15
    assert q[6:] == [8] * 26
    # positive extreme m = +4: d = -0.5, so m comes back as -0.5 * (0 - 8)
    w = np.zeros(32, np.float32)
    w[0], w[17] = 4.0, -1.0
    blk = oracle.quantize(Q4_0, w, 1, 32)
    assert blk[:2].view(np.uint16)[0] == 0xB800  # -0.5
    assert blk[2] & 15 == 0 and blk[2 + 1] >> 4 == 10  # -1 / -0.5 = 2 -> q = 10
    # ties between +a and -a: the first element decides the sign of d
    w = np.zeros(32, np.float32)
    w[3], w[9] = -2.0, 2.0
    assert oracle.quantize(Q4_0, w, 1, 32)[:2].view(np.uint16)[0] == half_bits(0.25)


def test_zero_block_and_tiny_scales():
    z = np.zeros((2, 64), np.float32)
    q4 = oracle.quantize(Q4_0, z, 2, 64)
    assert (q4.reshape(4, 18)[:, :2] == 0).all() and (q4.reshape(4, 18)[:, 2:] == 0x88).all()
    assert (oracle.quantize(I8_B64, z, 2, 64) == 0).all()
    # max |w| / 127 below half the smallest subnormal: d = +0, every q = 0
    w = np.zeros(32, np.float32)
    w[0] = 127 * 2.0 ** -26
    assert (oracle.quantize(Q8_0, w, 1, 32) == 0).all()


def test_rejects():
    w = np.ones((1, 32), np.float32)
    w[0, 5] = np.nan
    for fmt in (Q4_0, Q8_0):
        with pytest.raises(ValueError):
            oracle.quantize(fmt, w, 1, 32)
    big = np.full((1, 32), 127 * 65520.0, np.float32)  # scale past 65504
    with pytest.raises(ValueError):
        oracle.quantize(Q8_0, big, 1, 32)
    with pytest.raises(ValueError):
        oracle.quantize(3, np.ones((1, 256), np.float32), 1, 256)  # no Q6_K quantizer


def _codes(fmt, blk, be):
    d = oracle.fp16_to_double(int(blk[:2].view(np.uint16)[0]))
    if fmt == Q4_0:
        q = np.array([(blk[2 + j] & 15) if j < 16 else (blk[2 + j - 16] >> 4) for j in range(be)])
        return d, q.astype(np.int64) - 8, np.arange(-8, 8)
    return d, blk[2:2 + be].view(np.int8).astype(np.int64), np.arange(-127, 128)


@pytest.mark.parametrize("fmt,be", [(Q4_0, 32), (Q8_0, 32), (I8_B64, 64)])
def test_each_code_is_the_nearest(fmt, be):
    """Brute force: given the block's scale, every stored code is a nearest
    code to its weight, and on a tie the one farther from zero; the scale is
    the binary16 nearest to max|w|/127 (int8) or m/-8 (Q4_0)."""
    rng = np.random.default_rng(fmt)
    for t in range(300):
        w = (rng.standard_normal(be) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        if t % 5 == 0:  # exact half-way cases: integers and half-integers times a power of two
            w = (rng.integers(-40, 41, be) / 2.0 * 2.0 ** rng.integers(-8, 4)).astype(np.float32)
        blk = oracle.quantize(fmt, w, 1, be)
        d, q, cand = _codes(fmt, blk, be)
        wd = w.astype(np.float64)
        want = half_bits(wd[np.argmax(np.abs(wd))] / -8.0) if fmt == Q4_0 else \
            half_bits(np.abs(wd).max() / 127.0)
        if want & 0x7fff == 0:  # the scale rounds to zero: stored as +0, every value 0
            assert blk[:2].view(np.uint16)[0] == 0 and (q == 0).all()
            continue
        assert blk[:2].view(np.uint16)[0] == want
        for j in range(be):
            err = np.abs(wd[j] - d * cand)
            best = err.min()
            ties = cand[err == best]
            assert abs(wd[j] - d * q[j]) == best, (t, j)
            assert q[j] == ties[np.argmax(np.abs(ties))], (t, j)


@pytest.mark.parametrize("fmt,be", [(Q4_0, 32), (Q8_0, 32), (I8_B64, 64)])
def test_round_trip_error_bound(fmt, be):
    """Dequantized by the pinned decoder, every weight is within half a step
    of its input, except Q4_0 weights past +7.5 steps (clamped to 15)."""
    rng = np.random.default_rng(10 + fmt)
    N, K = 7, 4 * be
    w = rng.standard_normal((N, K)).astype(np.float32) * 0.05
    canon = oracle.quantize(fmt, w, N, K)
    back = oracle.dequant(fmt, canon, N, K)
    d = np.array([oracle.fp16_to_double(int(v)) for v in
                  canon.reshape(-1, oracle.block_bytes(fmt))[:, :2].copy().view(np.uint16)[:, 0]])
    d = np.repeat(np.abs(d), be).reshape(N, K)
    err = np.abs(back - w.astype(np.float64))
    if fmt == Q4_0:
        ok = err <= d / 2 + 1e-300
        clamped = ~ok
        assert (err[clamped] <= d[clamped] * (1 + 2.0 ** -10)).all()  # the +8 side of m's block
    else:
        # |w| / d may exceed 127.5 by the scale's rounding only: error within 127 d 2^-11
        assert (err <= d / 2 + 127 * d * 2.0 ** -11).all()
