"""Host quantizer (lean_quantize, include/lean_quant.h) against the oracle's
quantizer, byte for byte (CPU; no GPU involved).  The oracle's quantizer is
pinned in test_oracle_quant_pins.py."""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import build as lib_build
from block_quantized_weight_dot_gb300 import synthetic as syn

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


@pytest.fixture(scope="module")
def lean():
    lib_build.build()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def inputs(rng, N, K, kind):
    if kind == "normal":
        return (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    if kind == "wide":  # every row its own magnitude, from binary16-subnormal scales up
        return (rng.standard_normal((N, K)) * 10.0 ** rng.uniform(-9, 5, (N, 1))).astype(np.float32)
    if kind == "halves":  # many exact half-way quotients
        return (rng.integers(-64, 65, (N, K)) / 4.0 * 2.0 ** rng.integers(-6, 6, (N, 1))).astype(np.float32)
    if kind == "sparse":  # zero blocks and single spikes
        w = np.zeros((N, K), np.float32)
        idx = rng.random((N, K)) < 0.05
        w[idx] = rng.standard_normal(idx.sum()).astype(np.float32) * 3
        return w
    raise ValueError(kind)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("kind", ["normal", "wide", "halves", "sparse"])
def test_matches_oracle_bytes(lean, fmt, kind):
    rng = np.random.default_rng((fmt, len(kind)))
    be = syn.BLOCK_ELEMS[fmt]
    for N, K in ((1, be), (37, 5 * be), (64, 32 * be)):
        w = inputs(rng, N, K, kind)
        got = lean.lean_quantize(fmt, w, N, K)
        want = oracle.quantize(fmt, w, N, K)
        assert got.tobytes() == want.tobytes(), (kind, N, K)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_threads_do_not_change_bytes(lean, fmt):
    rng = np.random.default_rng(3)
    be = syn.BLOCK_ELEMS[fmt]
    w = inputs(rng, 203, 8 * be, "wide")
    one = lean.lean_quantize(fmt, w, 203, 8 * be, threads=1)
    for t in (0, 2, 7, 500):
        assert lean.lean_quantize(fmt, w, 203, 8 * be, threads=t).tobytes() == one.tobytes()


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_pack_round_trip_and_dequant(lean, fmt):
    """Quantized blocks go through lean_pack / lean_unpack_canonical unchanged,
    and decode (oracle) to within half a step of the input."""
    rng = np.random.default_rng(4)
    be = syn.BLOCK_ELEMS[fmt]
    N, K = 70, 6 * be
    w = inputs(rng, N, K, "normal")
    canon = lean.lean_quantize(fmt, w, N, K)
    assert lean.lean_unpack_canonical(fmt, lean.lean_pack(fmt, canon, N, K), N, K).tobytes() \
        == canon.tobytes()
    back = oracle.dequant(fmt, canon, N, K)
    amax = np.abs(w.reshape(N, K // be, be)).max(axis=2, keepdims=True)
    step = (amax / (8.0 if fmt == syn.Q4_0 else 127.0)).repeat(be, axis=2).reshape(N, K)
    assert (np.abs(back - w) <= step * (1 + 2.0 ** -9)).all()


def test_errors(lean):
    w = np.ones((2, 64), np.float32)
    f = lean._lib.lean_quantize
    buf = np.zeros(4096, np.uint8)
    assert f(syn.Q6_K, w.ctypes.data, buf.ctypes.data, 1, 256, 0) == lean.LEAN_ERR_FORMAT
    assert f(9, w.ctypes.data, buf.ctypes.data, 2, 64, 0) == lean.LEAN_ERR_FORMAT
    assert f(syn.Q8_0, None, buf.ctypes.data, 2, 64, 0) == lean.LEAN_ERR_NULL
    assert f(syn.Q8_0, w.ctypes.data, None, 2, 64, 0) == lean.LEAN_ERR_NULL
    assert f(syn.Q8_0, w.ctypes.data, buf.ctypes.data, 2, 63, 0) == lean.LEAN_ERR_SHAPE
    assert f(syn.I8_B64, w.ctypes.data, buf.ctypes.data, 0, 64, 0) == lean.LEAN_ERR_SHAPE
    assert f(syn.Q8_0, w.ctypes.data, buf.ctypes.data, 2, 64, -1) == lean.LEAN_ERR_SHAPE
    bad = w.copy()
    bad[1, 7] = np.inf
    assert f(syn.Q4_0, bad.ctypes.data, buf.ctypes.data, 2, 64, 0) == lean.LEAN_ERR_SHAPE
    big = np.full((1, 32), 3.0e38, np.float32)  # max|w| / 127 past 65504
    assert f(syn.Q8_0, big.ctypes.data, buf.ctypes.data, 1, 32, 1) == lean.LEAN_ERR_SHAPE
    with pytest.raises(lean.LeanError):
        lean.lean_quantize(syn.Q8_0, np.ones((2, 63), np.float32), 2, 63)


def test_any_finite_block_matches_oracle(lean):
    """Property: for any finite float32 block the product and the oracle agree
    byte for byte, or both refuse it (a scale past 65504)."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    floats = st.floats(allow_nan=False, allow_infinity=False, width=32)

    @hyp.settings(max_examples=300, deadline=None)
    @hyp.given(fmt=st.sampled_from(FMTS), data=st.data())
    def check(fmt, data):
        be = syn.BLOCK_ELEMS[fmt]
        w = np.array(data.draw(st.lists(floats, min_size=be, max_size=be)), np.float32)
        try:
            want = oracle.quantize(fmt, w, 1, be)
        except ValueError:
            want = None
        if want is None:
            with pytest.raises(lean.LeanError):
                lean.lean_quantize(fmt, w, 1, be)
        else:
            assert lean.lean_quantize(fmt, w, 1, be).tobytes() == want.tobytes()

    check()
