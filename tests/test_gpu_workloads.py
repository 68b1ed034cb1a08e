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


def test_decode_stack_batch_x_planes():
    """The whole 32-layer decode step (224 GEMVs, 177 MB of Q4_0 weights) as
    one lean_qmatmul_batch call with a workspace, the launch the benchmark
    times: at this size x goes in as integer planes; every output of every
    linear against the oracle."""
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    stack = syn.smollm2_360m_decode_stack()
    items, keep, refs = [], [], []
    for lin in stack.linears:
        W, x = lin.make()
        Wd = lean.upload_packed(lin.fmt, W, lin.N, lin.K)
        xd = torch.from_numpy(np.ascontiguousarray(x.reshape(-1))).cuda()
        yd = torch.full((lin.N,), float("nan"), device="cuda")
        keep += [Wd, xd, yd]
        items.append((Wd, xd, yd, lin.N, lin.K))
        refs.append(oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K, threads=THREADS))
    probs = lean.make_problems(items)
    nb = lean.lean_batch_workspace_bytes(syn.Q4_0, probs)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    outs = []
    for rep in range(2):
        for it in items:
            it[2].fill_(float("nan"))
        lean.lean_qmatmul_batch(syn.Q4_0, probs, lean.LEAN_FLAG_EARLY_WEIGHTS, ws, nb)
        torch.cuda.synchronize()
        ys = [it[2].cpu().numpy().astype(np.float64) for it in items]
        for lin, y, (y_ref, bound) in zip(stack.linears, ys, refs):
            check_close(y[None, :], y_ref, bound, "stack " + lin.name)
        outs.append(ys)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    assert lean.lean_device_error(True) == 0


def test_decode_stack_batch_host_buffers():
    """The same decode step with x and y in pinned host memory, passed to the
    call as they are (the x-plane path reads x and writes y with plain loads
    and stores, across the host link): every output against the oracle, and
    bit for bit what device buffers give."""
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    stack = syn.smollm2_360m_decode_stack()
    dev, host, keep, refs = [], [], [], []
    for lin in stack.linears:
        W, x = lin.make()
        Wd = lean.upload_packed(lin.fmt, W, lin.N, lin.K)
        xh = torch.from_numpy(np.ascontiguousarray(x.reshape(-1))).pin_memory()
        yh = torch.full((lin.N,), float("nan")).pin_memory()
        xd, yd = xh.cuda(), torch.full((lin.N,), float("nan"), device="cuda")
        keep += [Wd, xh, yh, xd, yd]
        host.append((Wd, xh, yh, lin.N, lin.K))
        dev.append((Wd, xd, yd, lin.N, lin.K))
        refs.append(oracle.qmatmul(lin.fmt, W, x, lin.N, lin.K, threads=THREADS))
    nb = lean.lean_batch_workspace_bytes(syn.Q4_0, lean.make_problems(dev))
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS | lean.LEAN_FLAG_X_PLANES
    for items in (host, dev):
        lean.lean_qmatmul_batch(syn.Q4_0, lean.make_problems(items), flags, ws, nb)
    torch.cuda.synchronize()
    for lin, h, d, (y_ref, bound) in zip(stack.linears, host, dev, refs):
        yh = h[2].numpy().astype(np.float64)
        check_close(yh[None, :], y_ref, bound, "host buffers " + lin.name)
        assert np.array_equal(yh, d[2].cpu().numpy().astype(np.float64)), lin.name
    assert lean.lean_device_error(True) == 0


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
