"""The tolerance check discriminates: negative controls for the parity bar.

The parity bar is |y - y_ref| <= 1e-4 * sum_k |w x| + 1e-6 per output.  These
CPU tests show what that bar rejects, using the oracle as the reference:

  - a product whose weights (or activations) are rounded once to bf16, the
    plain tensor-core shortcut, fails it: on ~14% of outputs at K = 2048 with
    N(0,1) activations, on most outputs at K = 32, on every output whose
    activations carry the signs of the weights' rounding errors, and on a
    one-hot activation (a single product);
  - at K = 11008 (the Qwen2.5-3B down projection) the same shortcut passes on
    N(0,1) activations: the rounding errors of 11008 products mostly cancel,
    so the average case alone would not reject it.  The worst case still
    does, which is why the tensor-core path splits both operands into bf16
    pairs (three MMAs) instead of rounding them once;
  - that split (w = w_hi + w_lo, x = x_hi + x_lo, dropping w_lo * x_lo)
    passes every one of these cases with a wide margin.

The GPU paths themselves are held to the bar by the -m gpu tests; this file
only shows the bar has teeth.  The pages' GPU GEMMs dequantize to f32 for the
same reason ("oxinfer" crate page, Platforms and accelerators).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn

REL, ABS = 1e-4, 1e-6


def bf16(a):
    """fp32 -> the nearest bfloat16 (ties to even), as fp32."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def split_bf16(a):
    a = np.asarray(a, np.float32)
    hi = bf16(a)
    return hi, bf16(a - hi)  # a - hi is exact in fp32


def err_over_tol(y, y_ref, bound):
    return np.abs(np.asarray(y, np.float64) - y_ref) / (REL * bound + ABS)


def products(w, x):
    """(bf16 w, fp32 x), (fp32 w, bf16 x) and split-bf16 products, in fp64."""
    w = np.asarray(w, np.float32)
    x = np.asarray(x, np.float32)
    f = lambda a: np.asarray(a, np.float64)
    y_wb = f(x) @ f(bf16(w)).T
    y_xb = f(bf16(x)) @ f(w).T
    wh, wl = split_bf16(w)
    xh, xl = split_bf16(x)
    y_split = f(xh) @ f(wh).T + f(xl) @ f(wh).T + f(xh) @ f(wl).T
    return y_wb, y_xb, y_split


def ffn_rows(idx, rows):
    """The first `rows` rows of a Qwen2.5-3B FFN linear (Q4_0, seeded as in
    the workload), its M = 4 activations, and its exact weights."""
    lin = syn.qwen25_3b_ffn(4).linears[idx]
    W, x = lin.make()
    W = np.ascontiguousarray(W[:rows])
    return lin, W, x, oracle.dequant(lin.fmt, W, rows, lin.K).astype(np.float32)


def test_bf16_weights_fail_at_k2048():
    lin, W, x, w = ffn_rows(0, 512)  # 11008 x 2048: K = 2048
    y_ref, bound = oracle.qmatmul(lin.fmt, W, x, 512, lin.K)
    y_wb, y_xb, y_split = products(w, x)
    assert np.mean(err_over_tol(y_wb, y_ref, bound) > 1) > 0.05
    assert np.mean(err_over_tol(y_xb, y_ref, bound) > 1) > 0.05
    assert np.max(err_over_tol(y_split, y_ref, bound)) < 0.05


def test_bf16_passes_average_but_not_worst_case_at_k11008():
    lin, W, x, w = ffn_rows(1, 128)  # 2048 x 11008: K = 11008
    y_ref, bound = oracle.qmatmul(lin.fmt, W, x, 128, lin.K)
    y_wb, _, y_split = products(w, x)
    # average case: the rounding errors cancel, the shortcut gets through
    assert np.mean(err_over_tol(y_wb, y_ref, bound) > 1) < 0.01
    assert np.max(err_over_tol(y_split, y_ref, bound)) < 0.05
    # worst case: activations with the signs of each row's weight rounding errors
    rng = np.random.default_rng(71)
    rows = np.arange(32)
    sgn = np.where(w[rows] - bf16(w[rows]) >= 0, 1.0, -1.0)
    xa = (np.abs(rng.standard_normal((len(rows), lin.K))) * sgn).astype(np.float32)
    y_ref, bound = oracle.qmatmul_pairs(lin.fmt, W, xa, 128, lin.K, rows, rows)
    got_wb = np.array([np.float64(xa[i]) @ np.float64(bf16(w[r])) for i, r in enumerate(rows)])
    wh, wl = split_bf16(w[rows])
    xh, xl = split_bf16(xa)
    got_split = np.array([np.float64(xh[i]) @ np.float64(wh[i]) + np.float64(xl[i]) @ np.float64(wh[i])
                          + np.float64(xh[i]) @ np.float64(wl[i]) for i in range(len(rows))])
    r = err_over_tol(got_wb, y_ref, bound)
    assert np.all(r > 5), r.min()
    assert np.max(err_over_tol(got_split, y_ref, bound)) < 0.05


def test_bf16_weights_fail_one_hot():
    """x = e_k: y is the single weight w[n, k]; bf16 rounding of w is caught
    wherever it changes w by more than 1e-4 of itself (and 1e-6)."""
    lin, W, _, w = ffn_rows(0, 256)
    ks = [0, 1, 17, 31, 1000, 2047]
    x = np.zeros((len(ks), lin.K), np.float32)
    x[np.arange(len(ks)), ks] = 1.0
    y_ref, bound = oracle.qmatmul(lin.fmt, W, x, 256, lin.K)
    y_wb, _, y_split = products(w, x)
    assert np.mean(err_over_tol(y_wb, y_ref, bound) > 1) > 0.3
    assert np.array_equal(y_split, y_ref)  # the Q4_0 weight split is exact


@pytest.mark.parametrize("fmt", [syn.Q4_0, syn.Q8_0, syn.I8_B64, syn.Q6_K],
                         ids=["q4_0", "q8_0", "i8_b64", "q6_k"])
def test_small_k_and_split_margin(fmt):
    """One block along K: the shortcut fails on most outputs; the split bf16
    product stays far inside the bar for every format."""
    be = syn.BLOCK_ELEMS[fmt]
    N = 1024
    W, x = syn.make_problem(fmt, N, be, 4, seed=(72, fmt))
    w = oracle.dequant(fmt, W, N, be).astype(np.float32)
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, be)
    y_wb, y_xb, y_split = products(w, x)
    if be == 32:
        assert np.mean(err_over_tol(y_wb, y_ref, bound) > 1) > 0.5
        assert np.mean(err_over_tol(y_xb, y_ref, bound) > 1) > 0.5
    else:
        assert np.mean(err_over_tol(y_wb, y_ref, bound) > 1) > 0.2
    assert np.max(err_over_tol(y_split, y_ref, bound)) < 0.1
