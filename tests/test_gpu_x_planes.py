"""GPU parity of the x-plane (dp4a) path on activations that stress a block
floating-point encoding of x: outlier channels far above their neighbours,
outliers whose weights are zero, blocks of +-max next to tiny values, tiny
values that the encoding holds exactly, subnormals, values near the top of
the fp32 range, and Inf / NaN.

Activations of real models carry a few channels at 10^2..10^4 times the
median; a plane encoding with one scale per 32 elements would round the small
neighbours of such a channel to nothing.  Every case here runs the product with
LEAN_FLAG_X_PLANES and a workspace (the path a decode step takes), once as a
single call and once as part of a batch, and is compared element by element
with the fp64 oracle under |y - y_ref| <= 1e-4 * sum|w x| + 1e-6.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]
N, K = 300, 2048


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def zero_weight(fmt, W, ks):
    """Canonical blocks with the weight of every row at columns ks set to 0
    (Q4_0: q = 8; the int8 formats: q = 0)."""
    be, bb = syn.BLOCK_ELEMS[fmt], syn.BLOCK_BYTES[fmt]
    W = W.copy().reshape(W.shape[0], -1, bb)
    for k in ks:
        b, j = divmod(int(k), be)
        if fmt == syn.Q4_0:
            if j < 16:
                W[:, b, 2 + j] = (W[:, b, 2 + j] & 0xF0) | 0x08
            else:
                W[:, b, 2 + j - 16] = (W[:, b, 2 + j - 16] & 0x0F) | 0x80
        else:
            W[:, b, 2 + j] = 0
    return W.reshape(W.shape[0], -1)


def run_planes(lean, fmt, W, x, n, k, batch):
    """y of the x-plane path: lean_qmatmul_ws (batch=False) or the problem as
    the middle one of three in lean_qmatmul_batch (batch=True)."""
    torch = torch_cuda()
    Wd = lean.upload_packed(fmt, W, n, k)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32).reshape(-1)).cuda()
    yd = torch.full((n,), float("nan"), device="cuda")
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS | lean.LEAN_FLAG_X_PLANES
    if not batch:
        nb = lean.lean_qmatmul_workspace_bytes(fmt, n, k, 1)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        lean.lean_qmatmul_ws(fmt, Wd, xd, yd, n, k, 1, flags, ws, nb)
    else:
        others = []
        for i in range(2):
            Wo, xo = syn.make_problem(fmt, 64, k, 1, seed=(50, fmt, i))
            others.append((lean.upload_packed(fmt, Wo, 64, k), torch.from_numpy(xo.reshape(-1)).cuda(),
                           torch.empty(64, device="cuda"), 64, k))
        probs = lean.make_problems([others[0], (Wd, xd, yd, n, k), others[1]])
        nb = lean.lean_batch_workspace_bytes(fmt, probs)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        lean.lean_qmatmul_batch(fmt, probs, flags, ws, nb)
    torch.cuda.synchronize()
    assert lean.lean_device_error(True) == 0
    return yd.cpu().numpy().astype(np.float64)[None, :]


def outlier_x(rng, amp, sign=1.0, every=1):
    """N(0,1) x with element 5 of every `every`-th 32-block set to sign * amp."""
    x = rng.standard_normal(K).astype(np.float32)
    pos = np.arange(0, K, 32 * every) + 5
    x[pos] = np.float32(sign * amp)
    return x, pos


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("amp", [1e2, 1e3, 1e4, 1e5])
@pytest.mark.parametrize("zeroed", [False, True], ids=["w", "w0"])
@pytest.mark.parametrize("batch", [False, True], ids=["single", "batch"])
def test_outlier_channels(lean, fmt, amp, zeroed, batch):
    """One element per 32-block at amp times an N(0,1) background, of both
    signs (alternating rows of blocks), with and without zero weights on it."""
    rng = np.random.default_rng((51, fmt, int(amp)))
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(52, fmt))
    x, pos = outlier_x(rng, amp)
    x[pos[1::2]] *= -1
    if zeroed:
        W = zero_weight(fmt, W, pos)
    y = run_planes(lean, fmt, W, x, N, K, batch)
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
    check_close(y, y_ref, bound, "%s amp=%g zeroed=%d" % (syn.FORMAT_NAMES[fmt], amp, zeroed))


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_sparse_outliers(lean, fmt):
    """Outliers in a few blocks only (the rest plain N(0,1)): the marked
    blocks take the exact path, the others the planes, in one call."""
    rng = np.random.default_rng((53, fmt))
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(54, fmt))
    x, pos = outlier_x(rng, 3e4, sign=-1.0, every=7)
    W = zero_weight(fmt, W, pos)
    for batch in (False, True):
        y = run_planes(lean, fmt, W, x, N, K, batch)
        y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
        check_close(y, y_ref, bound, "sparse outliers batch=%d" % batch)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_max_next_to_tiny(lean, fmt):
    """Blocks of +-max in half the elements and tiny values in the other
    half; rows whose only nonzero weights sit on the tiny values (the worst
    case for a shared scale: the whole result comes from the tiny elements)."""
    rng = np.random.default_rng((55, fmt))
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(56, fmt))
    x = np.empty(K, np.float32)
    big = np.arange(K) % 2 == 0
    x[big] = np.where(rng.random(big.sum()) < 0.5, -1e4, 1e4).astype(np.float32)
    x[~big] = (rng.standard_normal((~big).sum()) * 1e-3).astype(np.float32)
    # the first 100 rows weigh only the tiny elements
    Wz = zero_weight(fmt, W, np.flatnonzero(big))
    W = np.concatenate([Wz[:100], W[100:]])
    for batch in (False, True):
        y = run_planes(lean, fmt, W, x, N, K, batch)
        y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
        check_close(y, y_ref, bound, "max next to tiny batch=%d" % batch)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_tiny_exact_neighbours(lean, fmt):
    """Blocks whose elements are the largest one and exact small multiples of
    its quantum (the encoding holds them exactly, so the block keeps the
    plane path): negative ones have small digits only in balanced form, and
    the weight of the large element is zero, so the tiny ones make y."""
    rng = np.random.default_rng((57, fmt))
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(58, fmt))
    x = np.empty(K, np.float32)
    x[:] = -np.ldexp(rng.integers(1, 4, K).astype(np.float32), -29)  # -q, -2q, -3q
    pos = np.arange(0, K, 32) + 11
    x[pos] = 1.0  # max of every block: X = 2^29 scaled
    W = zero_weight(fmt, W, pos)
    for batch in (False, True):
        y = run_planes(lean, fmt, W, x, N, K, batch)
        y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
        check_close(y, y_ref, bound, "tiny exact neighbours batch=%d" % batch)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_extreme_ranges(lean, fmt):
    """Blocks of subnormals, of zeros, of values near 1e38 and of mixed
    exponents across the whole fp32 range, side by side."""
    rng = np.random.default_rng((59, fmt))
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(60, fmt))
    nb = K // 32
    x = rng.standard_normal(K).astype(np.float32)
    xb = x.reshape(nb, 32)
    xb[0::5] *= np.float32(1e-41)   # subnormals
    xb[1::5] = 0.0
    xb[2::5] *= np.float32(1e36)    # near the top (|w x| stays finite)
    xb[3::5] *= np.ldexp(np.float32(1), rng.integers(-60, 60, (len(xb[3::5]), 32))).astype(np.float32)
    for batch in (False, True):
        y = run_planes(lean, fmt, W, x, N, K, batch)
        y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
        assert np.all(np.isfinite(y_ref))
        check_close(y, y_ref, bound, "extreme ranges batch=%d" % batch)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_inf_nan_propagate(lean, fmt):
    """An Inf or NaN in x gives what IEEE arithmetic gives in the oracle: NaN
    where it does (0 * Inf, Inf - Inf, anything * NaN), +-Inf otherwise."""
    W, x = syn.make_problem(fmt, N, K, 1, seed=(61, fmt))
    x = x.reshape(-1).copy()
    x[37] = np.inf
    x[1000] = np.nan
    y = run_planes(lean, fmt, W, x, N, K, False)
    y_ref, _ = oracle.qmatmul(fmt, W, x, N, K)
    assert np.array_equal(np.isnan(y), np.isnan(y_ref))
    x[1000] = 1.0
    Wz = zero_weight(fmt, W, [37])
    W2 = np.concatenate([Wz[:10], W[10:]])  # rows 0..9: 0 * Inf = NaN
    y = run_planes(lean, fmt, W2, x, N, K, False)
    y_ref, bound = oracle.qmatmul(fmt, W2, x, N, K)
    assert np.array_equal(np.isnan(y), np.isnan(y_ref))
    fin = np.isfinite(y_ref)
    assert np.array_equal(y[~fin & ~np.isnan(y_ref)], y_ref[~fin & ~np.isnan(y_ref)])
    assert not fin.all()
