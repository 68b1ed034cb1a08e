"""Pins for the CPU oracle, independent of the oracle's own code.

Each test fixes the oracle to something other than itself: the IEEE binary16
definition (checked against numpy's own fp16 decoder), closed forms of
hand-built blocks (the Q4_0 example "all q = 9 times a ones vector gives K*d"),
per-element encoders written here from the block layouts (the oracle decodes;
these encode), exact integer products checked with numpy's matmul, invariants
(exact power-of-two scaling), the bytes-per-weight figures the "oxinfer" crate
page quotes (Performance), and brute force on tiny shapes.

Formats and their sources:
  Q4_0: "oxinfer" crate page, How it works (quant.rs): two nibbles per byte,
        f16 scale per 32 weights; value d*(q-8).
  Q8_0: "lean" README model table / parity tests (Q8_0 GGUF); 32 int8 + scale.
  INT8-B64: "wgpu-llm" README, INT8 mode: symmetric INT8, block size 64.
  Q6_K: "lean" README model table (Q6_K embedding); super-block of 256.
"""
import os

import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn

Q4_0, Q8_0, I8_B64, Q6_K = oracle.Q4_0, oracle.Q8_0, oracle.I8_B64, oracle.Q6_K


# ---- encoders written from the canonical layouts (the inverse direction) ----

def f16_bits(v: float) -> int:
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def enc_q4_0(d_bits, q):
    """One Q4_0 block: q[32] in 0..15; element j<16 -> low nibble of byte j,
    element j+16 -> high nibble of byte j."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= 0 and q.max() <= 15
    qs = bytearray(16)
    for j in range(32):
        if j < 16:
            qs[j] |= int(q[j])
        else:
            qs[j - 16] |= int(q[j]) << 4
    return bytes([d_bits & 0xFF, d_bits >> 8]) + bytes(qs)


def enc_int8(d_bits, q, n):
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (n,) and q.min() >= -128 and q.max() <= 127
    return bytes([d_bits & 0xFF, d_bits >> 8]) + bytes(int(v) & 0xFF for v in q)


def enc_q6_k(d_bits, q, sc):
    """One Q6_K super-block from q[256] in 0..63 and sc[16] int8.

    Element e: half h = e // 128; inside the half, group g = (e % 128) // 32 and
    lane l = e % 32.  Its low 4 bits sit in nibble g // 2 of ql[64h + 32(g % 2) + l],
    its high 2 bits in bits 2g..2g+1 of qh[32h + l]; its scale is sc[e // 16]."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 63
    ql = bytearray(128)
    qh = bytearray(64)
    for h in range(2):
        for g in range(4):
            for l in range(32):
                v = int(q[128 * h + 32 * g + l])
                ql[64 * h + 32 * (g % 2) + l] |= (v & 0xF) << (4 * (g // 2))
                qh[32 * h + l] |= (v >> 4) << (2 * g)
    scb = bytes(int(s) & 0xFF for s in sc)
    return bytes(ql) + bytes(qh) + scb + bytes([d_bits & 0xFF, d_bits >> 8])


def mat(blocks_per_row):
    """Canonical matrix bytes from a list of rows, each a list of block bytes."""
    return np.frombuffer(b"".join(b"".join(r) for r in blocks_per_row), dtype=np.uint8).copy()


# ---- P2: fp16 decode, all 65536 patterns, vs numpy's own decoder ------------

def test_fp16_decode_exhaustive():
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(b) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero kept
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_fp16_subnormal_and_extremes():
    assert oracle.fp16_to_double(0x0001) == 2.0 ** -24
    assert oracle.fp16_to_double(0x03FF) == 1023 * 2.0 ** -24
    assert oracle.fp16_to_double(0x0400) == 2.0 ** -14
    assert oracle.fp16_to_double(0x7BFF) == 65504.0
    assert oracle.fp16_to_double(0x7C00) == np.inf
    assert oracle.fp16_to_double(0xFC00) == -np.inf


# ---- P1: closed forms ----------------------------------------------------------

@pytest.mark.parametrize("K", [32, 96, 960])
def test_q4_0_all_nine_times_ones_is_K_d(K):
    """All q = 9 blocks (w = d) times a ones vector gives K*d."""
    d = f16_bits(0.0123)
    row = [enc_q4_0(d, [9] * 32)] * (K // 32)
    W = mat([row, row])
    y, b = oracle.qmatmul(Q4_0, W, np.ones(K, np.float32), 2, K)
    dv = float(np.float16(0.0123))
    assert y[0, 0] == K * dv and y[0, 1] == K * dv
    assert b[0, 0] == K * dv


def test_q4_0_per_block_scales_and_offsets():
    K = 128
    rng = np.random.default_rng(7)
    ds = [f16_bits(v) for v in (0.5, -0.25, 3.0, 0.0078125)]
    x = rng.integers(-4, 5, K).astype(np.float32)
    # q = 8 everywhere: every weight is zero
    W = mat([[enc_q4_0(d, [8] * 32) for d in ds]])
    y, b = oracle.qmatmul(Q4_0, W, x, 1, K)
    assert y[0, 0] == 0.0 and b[0, 0] == 0.0
    # q = 0 everywhere: w = -8 d_b
    W = mat([[enc_q4_0(d, [0] * 32) for d in ds]])
    y, b = oracle.qmatmul(Q4_0, W, x, 1, K)
    dv = [float(np.array(d, np.uint16).view(np.float16)) for d in ds]
    expect = sum(-8 * dv[i] * float(x[32 * i:32 * i + 32].sum()) for i in range(4))
    assert y[0, 0] == expect
    assert b[0, 0] == sum(8 * abs(dv[i]) * float(np.abs(x[32 * i:32 * i + 32]).sum()) for i in range(4))
    # q = 15: w = 7 d_b
    W = mat([[enc_q4_0(d, [15] * 32) for d in ds]])
    y, _ = oracle.qmatmul(Q4_0, W, np.ones(K, np.float32), 1, K)
    assert y[0, 0] == sum(7 * 32 * v for v in dv)


@pytest.mark.parametrize("fmt,be", [(Q8_0, 32), (I8_B64, 64)])
def test_int8_closed_forms(fmt, be):
    K = 4 * be
    d = f16_bits(0.002)
    dv = float(np.float16(0.002))
    ones = np.ones(K, np.float32)
    for qv in (1, -1, 127, -127, -128):
        W = mat([[enc_int8(d, [qv] * be, be)] * 4])
        y, b = oracle.qmatmul(fmt, W, ones, 1, K)
        assert y[0, 0] == K * qv * dv
        assert b[0, 0] == K * abs(qv) * dv


def test_q6_k_closed_forms():
    d = f16_bits(0.001)
    dv = float(np.float16(0.001))
    ones = np.ones(256, np.float32)
    # q = 33, sc = 1: every weight is d
    W = mat([[enc_q6_k(d, [33] * 256, [1] * 16)]])
    y, _ = oracle.qmatmul(Q6_K, W, ones, 1, 256)
    assert y[0, 0] == 256 * dv
    # same block, spelled as raw bytes: ql nibbles 1, qh 2-bit fields 2
    raw = bytes([0x11] * 128) + bytes([0xAA] * 64) + bytes([1] * 16) + bytes([d & 0xFF, d >> 8])
    assert raw == enc_q6_k(d, [33] * 256, [1] * 16)
    # q = 0, sc = -32: the extreme product (-32)(-32) = 1024 per weight
    W = mat([[enc_q6_k(d, [0] * 256, [-32] * 16)]])
    y, _ = oracle.qmatmul(Q6_K, W, ones, 1, 256)
    assert y[0, 0] == 256 * 1024 * dv
    # q = 63, sc = -32: -31*32 per weight
    W = mat([[enc_q6_k(d, [63] * 256, [-32] * 16)]])
    y, _ = oracle.qmatmul(Q6_K, W, ones, 1, 256)
    assert y[0, 0] == 256 * (-31 * 32) * dv


# ---- P3-style element order: per-element encoders vs the oracle's decode ----

def test_q4_0_element_order():
    rng = np.random.default_rng(11)
    for _ in range(20):
        q = rng.integers(0, 16, 32)
        d = f16_bits(float(rng.uniform(-2, 2)))
        w = oracle.dequant(Q4_0, mat([[enc_q4_0(d, q)]]), 1, 32)[0]
        dv = float(np.array(d, np.uint16).view(np.float16))
        assert np.array_equal(w, dv * (q - 8).astype(np.float64))


@pytest.mark.parametrize("fmt,be", [(Q8_0, 32), (I8_B64, 64)])
def test_int8_element_order(fmt, be):
    rng = np.random.default_rng(12)
    for _ in range(20):
        q = rng.integers(-128, 128, be)
        d = f16_bits(float(rng.uniform(-1, 1)))
        w = oracle.dequant(fmt, mat([[enc_int8(d, q, be)]]), 1, be)[0]
        dv = float(np.array(d, np.uint16).view(np.float16))
        assert np.array_equal(w, dv * q.astype(np.float64))


def test_q6_k_element_order():
    rng = np.random.default_rng(13)
    for _ in range(10):
        q = rng.integers(0, 64, 256)
        sc = rng.integers(-32, 32, 16)
        d = f16_bits(float(rng.uniform(-0.01, 0.01)))
        w = oracle.dequant(Q6_K, mat([[enc_q6_k(d, q, sc)]]), 1, 256)[0]
        dv = float(np.array(d, np.uint16).view(np.float16))
        expect = dv * np.repeat(sc, 16).astype(np.float64) * (q - 32).astype(np.float64)
        assert np.array_equal(w, expect)


def test_q6_k_single_element_positions():
    """Each element set alone to q = 63 (others 32, i.e. zero) lands at its own k."""
    d = f16_bits(1.0)
    for e in (0, 1, 15, 16, 31, 32, 63, 64, 95, 96, 127, 128, 159, 191, 223, 255):
        q = np.full(256, 32)
        q[e] = 63
        w = oracle.dequant(Q6_K, mat([[enc_q6_k(d, q, [1] * 16)]]), 1, 256)[0]
        nz = np.nonzero(w)[0]
        assert list(nz) == [e] and w[e] == 31.0


# ---- exact integer products vs numpy matmul (transposed-operand check) -----

@pytest.mark.parametrize("fmt", [Q4_0, Q8_0, I8_B64, Q6_K])
def test_exact_integer_product_vs_numpy(fmt):
    rng = np.random.default_rng(100 + fmt)
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 5, 2 * be, 3
    one = f16_bits(1.0)
    rows, qmat = [], np.zeros((N, K), np.int64)
    for n in range(N):
        row = []
        for b in range(K // be):
            if fmt == Q4_0:
                q = rng.integers(0, 16, 32)
                row.append(enc_q4_0(one, q))
                qmat[n, 32 * b:32 * b + 32] = q - 8
            elif fmt == Q6_K:
                q = rng.integers(0, 64, 256)
                sc = rng.integers(-32, 32, 16)
                row.append(enc_q6_k(one, q, sc))
                qmat[n, 256 * b:256 * b + 256] = np.repeat(sc, 16) * (q - 32)
            else:
                q = rng.integers(-127, 128, be)
                row.append(enc_int8(one, q, be))
                qmat[n, be * b:be * b + be] = q
        rows.append(row)
    W = mat(rows)
    x = rng.integers(-50, 51, (M, K))
    y, b = oracle.qmatmul(fmt, W, x.astype(np.float32), N, K)
    assert np.array_equal(y, (x @ qmat.T).astype(np.float64))
    assert np.array_equal(b, (np.abs(x) @ np.abs(qmat).T).astype(np.float64))


# ---- brute force on tiny seeded problems -------------------------------------

@pytest.mark.parametrize("fmt", [Q4_0, Q8_0, I8_B64, Q6_K])
def test_brute_force_tiny(fmt):
    be = syn.BLOCK_ELEMS[fmt]
    for N, K, M in ((1, be, 1), (3, 2 * be, 2), (4, be, 3)):
        W, x = syn.make_problem(fmt, N, K, M, seed=(9, fmt, N, K))
        w = oracle.dequant(fmt, W, N, K)
        y, b = oracle.qmatmul(fmt, W, x, N, K)
        for m in range(M):
            for n in range(N):
                s = 0.0
                a = 0.0
                for k in range(K):
                    p = w[n, k] * float(x[m, k])
                    s += p
                    a += abs(p)
                assert y[m, n] == s and b[m, n] == a


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0, I8_B64, Q6_K])
def test_threads_and_pairs_agree(fmt):
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 37, 4 * be, 3
    W, x = syn.make_problem(fmt, N, K, M, seed=(10, fmt))
    y1, b1 = oracle.qmatmul(fmt, W, x, N, K, threads=1)
    y4, b4 = oracle.qmatmul(fmt, W, x, N, K, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(b1, b4)
    mi = np.array([0, 2, 1, 2]); ni = np.array([0, 36, 17, 5])
    yp, bp = oracle.qmatmul_pairs(fmt, W, x, N, K, mi, ni)
    assert np.array_equal(yp, y1[mi, ni]) and np.array_equal(bp, b1[mi, ni])


# ---- invariants -----------------------------------------------------------------

@pytest.mark.parametrize("fmt", [Q4_0, Q8_0, I8_B64, Q6_K])
def test_power_of_two_scaling_exact(fmt):
    be = syn.BLOCK_ELEMS[fmt]
    W, x = syn.make_problem(fmt, 8, 2 * be, 2, seed=(11, fmt))
    y, b = oracle.qmatmul(fmt, W, x, 8, 2 * be)
    for s in (-3, 5):
        ys, bs = oracle.qmatmul(fmt, W, x * np.float32(2.0 ** s), 8, 2 * be)
        assert np.array_equal(ys, y * 2.0 ** s) and np.array_equal(bs, b * 2.0 ** s)


def test_q8_sign_flip_negates():
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, 32)
    d = f16_bits(0.01)
    x = rng.standard_normal(32).astype(np.float32)
    y1, _ = oracle.qmatmul(Q8_0, mat([[enc_int8(d, q, 32)]]), x, 1, 32)
    y2, _ = oracle.qmatmul(Q8_0, mat([[enc_int8(d, -q, 32)]]), x, 1, 32)
    assert y1[0, 0] == -y2[0, 0]


def test_weights_exact_in_fp32():
    """Every decoded weight of the synthetic laws is exactly an fp32 value."""
    for fmt in (Q4_0, Q8_0, I8_B64, Q6_K):
        be = syn.BLOCK_ELEMS[fmt]
        W, _ = syn.make_problem(fmt, 16, 4 * be, 1, seed=(12, fmt))
        w = oracle.dequant(fmt, W, 16, 4 * be)
        assert np.array_equal(w.astype(np.float32).astype(np.float64), w)


# ---- P7: bytes per weight against the "oxinfer" crate page (Performance) ------

def _page_figures():
    """tests/golden/page_figures.txt: key = value lines, each citing its page."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_figures.txt")
    figs = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (t.strip() for t in line.split("="))
                figs[k] = float(v)
    return figs


def test_bytes_per_weight_match_quoted_ratios():
    """The pages' figures (tests/golden/page_figures.txt): Q8 cuts bytes per
    token by 1.8x and Q4 by 3.5x against bf16, Q8 = 32 weights per f32 scale,
    Q4_0 = two nibbles per byte + f16 scale per 32 ("oxinfer" crate page,
    Performance; How it works); INT8 blocks of 64 weights cut VRAM ~2x against
    bf16 ("wgpu-llm" README, INT8 mode).  Our Q4_0 block gives the Q4 figure;
    the Q8 figure follows from the same accounting with a 4-byte scale."""
    figs = _page_figures()
    q4 = oracle.block_bytes(Q4_0) / oracle.block_elems(Q4_0)
    assert q4 == 1 / figs["q4_nibbles_per_byte"] + 2 / 32
    assert int(2 / q4 * 10) == int(figs["q4_bytes_cut_vs_bf16"] * 10)  # 3.55..: "3.5x"
    q8_f32 = (oracle.block_elems(Q8_0) + 4) / figs["q8_weights_per_f32_scale"]
    assert round(2 / q8_f32, 1) == figs["q8_bytes_cut_vs_bf16"]
    assert oracle.block_elems(I8_B64) == figs["int8_block_size"]
    assert round(2 / (oracle.block_bytes(I8_B64) / oracle.block_elems(I8_B64))) == \
        figs["int8_vram_cut_vs_bf16"]
    assert oracle.block_bytes(I8_B64) == 66 and oracle.block_bytes(Q6_K) == 210
    for fmt in (Q4_0, Q8_0, I8_B64, Q6_K):
        assert oracle.block_bytes(fmt) == syn.BLOCK_BYTES[fmt]
        assert oracle.block_elems(fmt) == syn.BLOCK_ELEMS[fmt]