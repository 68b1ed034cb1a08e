"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses.  Outputs are compared with the oracle in full where the oracle
finishes in seconds, otherwise on sampled (m, n) pairs computed one by one.
"""
import os

import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, run_gpu, torch_cuda

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


def _full(lin):
    W, x = lin.make()
    y = run_gpu(lin.fmt, W, x, lin.N, lin.K)
    y_ref, bound = oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K, threads=THREADS)
    return check_close(y, y_ref, bound, lin.name)


def _sampled(lin, n_samples, seed):
    W, x = lin.make()
    y = run_gpu(lin.fmt, W, x, lin.N, lin.K)
    rng = np.random.default_rng(seed)
    mi = rng.integers(0, lin.M, n_samples)
    ni = rng.integers(0, lin.N, n_samples)
    # always include the first and last rows of every 32-row group edge
    mi = np.concatenate([mi, [0, lin.M - 1, 0, lin.M - 1]])
    ni = np.concatenate([ni, [0, lin.N - 1, lin.N - 1, 0]])
    y_ref, bound = oracle.qmatmul_pairs(lin.fmt, W, x, lin.N, lin.K, mi, ni)
    assert np.all(np.isfinite(y))
    return check_close(y[mi, ni], y_ref, bound, lin.name)


def test_q4_0_gemv_960():
    torch_cuda()
    for lin in syn.q4_0_gemv_960().linears:
        _full(lin)


def test_decode_stack_layers():
    """Every distinct SmolLM2-360M linear shape, first and last layer, full."""
    torch_cuda()
    stack = syn.smollm2_360m_decode_stack()
    for lin in stack.linears[:7] + stack.linears[-7:]:
        _full(lin)


@pytest.mark.parametrize("fmt", [syn.Q8_0, syn.I8_B64], ids=["q8_0", "i8_b64"])
def test_tinyllama_full(fmt):
    torch_cuda()
    for lin in syn.tinyllama_gemv(fmt).linears:
        _full(lin)


@pytest.mark.parametrize("M", syn.QWEN25_3B_FFN_BATCHES)
def test_qwen_ffn(M):
    torch_cuda()
    for lin in syn.qwen25_3b_ffn(M).linears:
        if M <= 16:
            _full(lin)
        else:
            _sampled(lin, 3000, seed=M)


def test_q6_k_lm_head_sampled():
    torch_cuda()
    (lin,) = syn.qwen25_3b_lm_head().linears
    _sampled(lin, 4000, seed=5)
