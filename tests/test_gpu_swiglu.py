"""GPU parity of lean_qmatmul_swiglu: the fused gate / up projections of a
decode layer's FFN with the SiLU(gate) * up epilogue (the input of the down
projection), against the oracle's composition (oracle.swiglu).

Tolerance, from the products' bar and the epilogue's fp32 arithmetic: with
T_g = 1e-4 * sum|w_g x| + 1e-6 and T_u likewise, |silu'| <= 1.1,
  |h - h_ref| <= 1.1 * T_g * (|u| + T_u) + |silu(g)| * T_u + 2^-20 |h| + 1e-12
(expf within 2 ulp, three more roundings).  Covered: the FFN shapes of
SmolLM2-360M, TinyLlama-1.1B and Qwen2.5-3B, every format, rows split over 1 to
4 CTAs per matrix (clusters of 2 to 8), ragged N, large activations (SiLU
saturating on both sides), the chain swiglu -> down with programmatic
dependent launch, and argument errors.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def check_h(h, fmt, Wg, Wu, x, N, K, what):
    h_ref, g, u, bg, bu = oracle.swiglu(fmt, Wg, Wu, x, N, K)
    tg, tu = 1e-4 * bg + 1e-6, 1e-4 * bu + 1e-6
    silu = g / (1.0 + np.exp(-g))
    lim = 1.1 * tg * (np.abs(u) + tu) + np.abs(silu) * tu + 2.0 ** -20 * np.abs(h_ref) + 1e-12
    err = np.abs(np.asarray(h, np.float64) - h_ref)
    bad = ~(err <= lim)
    assert not bad.any(), "%s: %d of %d out; first %d: h=%r ref=%r lim=%r" % (
        what, bad.sum(), N, np.argmax(bad), h[np.argmax(bad)], h_ref[np.argmax(bad)],
        lim[np.argmax(bad)])
    return h_ref


def run_swiglu(lean, fmt, Wg, Wu, x, N, K, flags=0):
    torch = torch_cuda()
    Wgd = lean.upload_packed(fmt, Wg, N, K)
    Wud = lean.upload_packed(fmt, Wu, N, K)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32).reshape(-1)).cuda()
    hd = torch.full((N + 32,), float("nan"), device="cuda")
    lean.lean_qmatmul_swiglu(fmt, Wgd, Wud, xd, hd, N, K, flags)
    torch.cuda.synchronize()
    h = hd.cpu().numpy().astype(np.float64)
    assert np.isnan(h[N:]).all()  # nothing written past h
    return h[:N]


CASES = [
    (syn.Q4_0, 2560, 960),     # SmolLM2-360M gate / up
    (syn.Q4_0, 11008, 2048),   # Qwen2.5-3B
    (syn.Q8_0, 5632, 2048),    # TinyLlama-1.1B
    (syn.I8_B64, 5632, 2048),
    (syn.Q6_K, 1000, 2048),
    (syn.Q4_0, 33, 64),        # ragged, short rows
    (syn.Q4_0, 100, 4096),     # 2 CTAs per matrix
    (syn.Q4_0, 70, 8192),      # 4 CTAs per matrix (a cluster of 8)
    (syn.Q8_0, 40, 4096),
]


@pytest.mark.parametrize("fmt,N,K", CASES)
def test_swiglu_parity(lean, fmt, N, K):
    Wg, x = syn.make_problem(fmt, N, K, 1, seed=(130, fmt, N, K))
    Wu, _ = syn.make_problem(fmt, N, K, 1, seed=(131, fmt, N, K))
    h = run_swiglu(lean, fmt, Wg, Wu, x, N, K)
    check_h(h, fmt, Wg, Wu, x, N, K, "%s %dx%d" % (syn.FORMAT_NAMES[fmt], N, K))
    h2 = run_swiglu(lean, fmt, Wg, Wu, x, N, K, flags=lean.LEAN_FLAG_EARLY_WEIGHTS)
    assert np.array_equal(h, h2)  # deterministic


def test_swiglu_saturating(lean):
    """Activations large enough that silu(g) is ~g for large g and ~0 for
    very negative g."""
    fmt, N, K = syn.Q4_0, 512, 960
    Wg, x = syn.make_problem(fmt, N, K, 1, seed=(132,))
    Wu, _ = syn.make_problem(fmt, N, K, 1, seed=(133,))
    x = x * np.float32(40.0)
    h = run_swiglu(lean, fmt, Wg, Wu, x, N, K)
    h_ref = check_h(h, fmt, Wg, Wu, x, N, K, "saturating")
    _, g, _, _, _ = oracle.swiglu(fmt, Wg, Wu, x, N, K)
    assert (g > 30).any() and (g < -30).any()


def test_swiglu_then_down_chain(lean):
    """swiglu -> down with programmatic dependent launch, repeated: down must
    read h only after swiglu wrote it (h starts as NaN each time)."""
    torch = torch_cuda()
    fmt, F, D = syn.Q4_0, 2560, 960
    Wg, x = syn.make_problem(fmt, F, D, 1, seed=(134,))
    Wu, _ = syn.make_problem(fmt, F, D, 1, seed=(135,))
    Wd, _ = syn.make_problem(fmt, D, F, 1, seed=(136,))
    Wgd, Wud, Wdd = (lean.upload_packed(fmt, W, n, k) for W, n, k in ((Wg, F, D), (Wu, F, D), (Wd, D, F)))
    xd = torch.from_numpy(x.reshape(-1)).cuda()
    s = torch.cuda.Stream()
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS
    outs = []
    for rep in range(3):
        hd = torch.full((F,), float("nan"), device="cuda")
        yd = torch.full((D,), float("nan"), device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            lean.lean_qmatmul_swiglu(fmt, Wgd, Wud, xd, hd, F, D, flags, s)
            lean.lean_qmatmul_ex(fmt, Wdd, hd, yd, D, F, 1, flags, s)
        s.synchronize()
        h = hd.cpu().numpy()
        check_h(h.astype(np.float64), fmt, Wg, Wu, x, F, D, "chain h")
        y_ref, bound = oracle.qmatmul(fmt, Wd, h, D, F)  # down applied to the GPU's h
        check_close(yd.cpu().numpy().astype(np.float64)[None, :], y_ref, bound, "chain down")
        outs.append(yd.cpu().numpy())
    assert all(np.array_equal(outs[0], o) for o in outs)


def test_swiglu_argument_errors(lean):
    torch = torch_cuda()
    W, x = syn.make_problem(syn.Q4_0, 64, 8256, 1, seed=(137,))
    Wd = lean.upload_packed(syn.Q4_0, W, 64, 8256)
    xd = torch.from_numpy(x.reshape(-1)).cuda()
    hd = torch.empty(64, device="cuda")
    f = lean._lib.lean_qmatmul_swiglu
    st = torch.cuda.current_stream().cuda_stream
    a = (Wd.data_ptr(), Wd.data_ptr(), xd.data_ptr(), hd.data_ptr())
    assert f(0, *a, 64, 8256, 0, st) == lean.LEAN_ERR_SHAPE      # K past 4 CTAs per matrix
    assert f(0, *a, 64, 8192, 4, st) == lean.LEAN_ERR_FORMAT     # a flag it does not take
    assert f(0, *a, 64, 8192, 0, st) == lean.LEAN_OK
    assert f(0, None, Wd.data_ptr(), xd.data_ptr(), hd.data_ptr(), 64, 8192, 0, st) == lean.LEAN_ERR_NULL
    torch.cuda.synchronize()
