"""GPU parity of the one-wave M = 1 kernel (qmm_gemv_kernel): every product
whose row groups fit the GPU at once takes it by default.

Covered: rows split over 1 to 8 CTAs of a cluster (K from one block to the
longest rows it takes), ragged N, every format, batches whose problems have
different K (one cluster size for all: short rows leave CTAs idle), results
equal within the tolerance to the streaming kernel's (LEAN_FLAG_STREAM) and
bit-identical run to run, nothing written outside y, and the products that
do not fit one wave (falling back to the streaming kernel).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64, syn.Q6_K]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]
NB = {syn.Q4_0: 8, syn.Q8_0: 4, syn.I8_B64: 2, syn.Q6_K: 1}  # blocks per warp, at most


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def run(lean, fmt, W, x, N, K, flags=0, canary=0):
    torch = torch_cuda()
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32).reshape(-1)).cuda()
    yd = torch.full((N + canary,), float("nan"), device="cuda")
    lean.lean_qmatmul_ex(fmt, Wd, xd, yd, N, K, 1, flags)
    torch.cuda.synchronize()
    out = yd.cpu().numpy().astype(np.float64)
    if canary:
        assert np.isnan(out[N:]).all()
    return out[None, :N]


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("cl", [1, 2, 3, 5, 8])
def test_cluster_splits(lean, fmt, cl):
    """K chosen so that the row needs exactly cl CTAs of 8 warps x NB blocks
    (the last one partly filled), N ragged."""
    be = syn.BLOCK_ELEMS[fmt]
    blocks = 8 * NB[fmt] * (cl - 1) + max(1, 3 * NB[fmt])
    N, K = 97, blocks * be
    W, x = syn.make_problem(fmt, N, K, 1, seed=(90, fmt, cl))
    y = run(lean, fmt, W, x, N, K, canary=64)
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=4)
    check_close(y, y_ref, bound, "%s cl=%d K=%d" % (syn.FORMAT_NAMES[fmt], cl, K))
    y2 = run(lean, fmt, W, x, N, K)
    assert np.array_equal(y, y2)
    ys = run(lean, fmt, W, x, N, K, flags=4)  # the streaming kernel
    check_close(ys, y_ref, bound, "stream")


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_mixed_k_batch(lean, fmt):
    """One launch for problems of different K and N (q/k/v-like and a long
    row), with and without programmatic dependent launch."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    shapes = [(960, 30 * be // 32), (320, 30 * be // 32), (64, 80 * be // 32), (5, 1), (33, 2)]
    if fmt == syn.Q6_K:
        shapes = [(N, max(1, nb // 8)) for N, nb in shapes]
    items, keep, refs = [], [], []
    for i, (N, nb) in enumerate(shapes):
        K = nb * be
        W, x = syn.make_problem(fmt, N, K, 1, seed=(91, fmt, i))
        Wd = lean.upload_packed(fmt, W, N, K)
        xd = torch.from_numpy(x.reshape(-1)).cuda()
        yd = torch.full((N,), float("nan"), device="cuda")
        keep += [Wd, xd, yd]
        items.append((Wd, xd, yd, N, K))
        refs.append(oracle.qmatmul(fmt, W, x, N, K))
    probs = lean.make_problems(items)
    for flags in (0, lean.LEAN_FLAG_EARLY_WEIGHTS):
        for it in items:
            it[2].fill_(float("nan"))
        lean.lean_qmatmul_batch(fmt, probs, flags, None, 0)
        torch.cuda.synchronize()
        for (Wd, xd, yd, N, K), (y_ref, bound) in zip(items, refs):
            check_close(yd.cpu().numpy().astype(np.float64)[None, :], y_ref, bound,
                        "mixed batch N=%d K=%d" % (N, K))


def test_workloads_on_the_one_wave_kernel(lean):
    """The single products of the benchmark's workloads that fit one wave."""
    lins = list(syn.q4_0_gemv_960().linears) + list(syn.smollm2_360m_decode_stack(1).linears) + \
        list(syn.tinyllama_gemv(syn.Q8_0).linears) + list(syn.qwen25_3b_ffn(1).linears)
    for lin in lins:
        W, x = lin.make()
        y = run(lean, lin.fmt, W, x, lin.N, lin.K)
        y_ref, bound = oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K, threads=8)
        check_close(y, y_ref, bound, lin.name)
