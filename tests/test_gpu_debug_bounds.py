"""Every kernel path through the LEAN_DEBUG build of the library, whose
kernels check each global-memory index against the buffers their arguments
describe and report one outside them as LEAN_ERR_KERNEL_BOUNDS (device error
bit 32) instead of touching it.

Small odd shapes (N = 1, 3, 33, 100; K of one block up to a few steps), so
that ragged row groups, partial steps and the smallest launches all run,
plus the larger tiles of the tensor-core paths: each product must match the
oracle and leave the device status at LEAN_OK.  A canary tail after y must
keep its NaNs.  Nothing here plants a bad index: a kernel that computed one
would be a bug, caught by the status check.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64, syn.Q6_K]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import build
    from block_quantized_weight_dot_gb300 import lean as L
    dbg = L.open_library(build.build(debug=True))
    prev = L.use_library(dbg)
    assert L.lean_debug_build() == 1
    assert L.lean_device_status(True) == L.LEAN_OK
    yield L
    L.use_library(prev)


def product(lean, fmt, N, K, M, flags=0, workspace=False, seed=0):
    torch = torch_cuda()
    W, x = syn.make_problem(fmt, N, K, M, seed=(90, fmt, N, K, M, seed))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32).reshape(-1)).cuda()
    tail = 64
    yb = torch.full((M * N + tail,), float("nan"), device="cuda")
    yd = yb[:M * N]
    if workspace:
        nb = max(lean.lean_qmatmul_workspace_bytes(fmt, N, K, M), 256)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        lean.lean_qmatmul_ws(fmt, Wd, xd, yd, N, K, M, flags, ws, nb)
    else:
        lean.lean_qmatmul_ex(fmt, Wd, xd, yd, N, K, M, flags)
    torch.cuda.synchronize()
    status = lean.lean_device_status(True)
    out = yb.cpu().numpy().astype(np.float64)
    assert np.isnan(out[M * N:]).all(), "write past the end of y"
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
    check_close(out[:M * N].reshape(M, N), y_ref, bound,
                "%s N=%d K=%d M=%d flags=%d ws=%s" % (syn.FORMAT_NAMES[fmt], N, K, M, flags, workspace))
    assert status == lean.LEAN_OK, lean.status_str(status)


def ks(fmt, nblocks):
    return syn.BLOCK_ELEMS[fmt] * nblocks


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("N", [1, 3, 33, 100])
def test_m1_paths(lean, fmt, N):
    for nb in (1, 3, 9):
        K = ks(fmt, nb)
        product(lean, fmt, N, K, 1)                                          # one-wave kernel
        product(lean, fmt, N, K, 1, flags=lean.LEAN_FLAG_STREAM)             # streaming ring
        product(lean, fmt, N, K, 1, workspace=True)                          # stream-K
        if fmt != syn.Q6_K:
            product(lean, fmt, N, K, 1, flags=lean.LEAN_FLAG_X_PLANES, workspace=True)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("M", [2, 5, 8, 15])
def test_small_m_paths(lean, fmt, M):
    for N, nb in ((1, 1), (33, 3), (100, 9)):
        product(lean, fmt, N, ks(fmt, nb), M)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("M", [16, 40, 70, 257])
def test_tensor_core_paths(lean, fmt, M):
    for N, nb in ((1, 1), (33, 3), (130, 9)):
        K = ks(fmt, nb)
        product(lean, fmt, N, K, M)
        product(lean, fmt, N, K, M, workspace=True)


def test_batch_embed_dequant_swiglu(lean):
    torch = torch_cuda()
    fmt = syn.Q4_0
    # batch of odd problems with the plane path
    items, refs = [], []
    for i, (N, nb) in enumerate(((1, 1), (3, 2), (33, 9), (100, 17))):
        K = ks(fmt, nb)
        W, x = syn.make_problem(fmt, N, K, 1, seed=(91, i))
        Wd = lean.upload_packed(fmt, W, N, K)
        xd = torch.from_numpy(x.reshape(-1)).cuda()
        yd = torch.full((N,), float("nan"), device="cuda")
        items.append((Wd, xd, yd, N, K))
        refs.append(oracle.qmatmul(fmt, W, x, N, K))
    probs = lean.make_problems(items)
    nb_ws = lean.lean_batch_workspace_bytes(fmt, probs)
    ws = torch.zeros(nb_ws, dtype=torch.uint8, device="cuda")
    lean.lean_qmatmul_batch(fmt, probs, lean.LEAN_FLAG_X_PLANES, ws, nb_ws)
    torch.cuda.synchronize()
    assert lean.lean_device_status(True) == lean.LEAN_OK
    for (Wd, xd, yd, N, K), (y_ref, bound) in zip(items, refs):
        check_close(yd.cpu().numpy()[None, :], y_ref, bound, "batch N=%d" % N)
    # embedding rows and dequantisation of a 33 x 3-block Q6_K table
    fmt6, N, K = syn.Q6_K, 33, ks(syn.Q6_K, 3)
    W, _ = syn.make_problem(fmt6, N, K, 1, seed=(92,))
    Wd = lean.upload_packed(fmt6, W, N, K)
    ids = torch.tensor([0, 32, 7, 7, 31], dtype=torch.int32, device="cuda")
    out = torch.empty((5, K), device="cuda")
    lean.lean_embed_rows(fmt6, Wd, ids, out, 5, N, K)
    wd = torch.empty((N, K), device="cuda")
    lean.lean_dequant(fmt6, Wd, wd, N, K)
    torch.cuda.synchronize()
    assert lean.lean_device_status(True) == lean.LEAN_OK
    w_ref = oracle.dequant(fmt6, W, N, K)
    assert np.array_equal(wd.cpu().numpy().astype(np.float64), w_ref)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), w_ref[[0, 32, 7, 7, 31]])
    # the fused gate / up with SiLU
    N, K = 33, ks(fmt, 9)
    Wg, x = syn.make_problem(fmt, N, K, 1, seed=(93, 0))
    Wu, _ = syn.make_problem(fmt, N, K, 1, seed=(93, 1))
    h = torch.full((N,), float("nan"), device="cuda")
    lean.lean_qmatmul_swiglu(fmt, lean.upload_packed(fmt, Wg, N, K), lean.upload_packed(fmt, Wu, N, K),
                             torch.from_numpy(x.reshape(-1)).cuda(), h, N, K)
    torch.cuda.synchronize()
    assert lean.lean_device_status(True) == lean.LEAN_OK
    assert np.isfinite(h.cpu().numpy()).all()


def test_status_of_other_device_errors(lean):
    """Bits other than the bounds bit map to LEAN_ERR_DEVICE: the documented
    ones that can be raised without a fault (an embedding id out of range,
    the bounded-wait self-test)."""
    torch = torch_cuda()
    fmt, N, K = syn.Q8_0, 4, 32
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(94,))
    Wd = lean.upload_packed(fmt, W, N, K)
    ids = torch.tensor([5], dtype=torch.int32, device="cuda")
    out = torch.empty((1, K), device="cuda")
    lean.lean_embed_rows(fmt, Wd, ids, out, 1, N, K)
    assert lean.lean_device_status(True) == lean.LEAN_ERR_DEVICE
    lean.lean_wait_selftest(1000)
    assert lean.lean_device_status(True) == lean.LEAN_ERR_DEVICE
    assert lean.lean_device_status(True) == lean.LEAN_OK
