"""The allocation-free M = 1 entry point, lean_qmatmul_fixed_ws.

It is for callers that cannot allocate device memory where they run the
product (stream capture, host frameworks that own the memory pool, loops that
must not risk the device synchronisation of cudaMalloc / cudaFree): its
scratch is a fixed array inside the library.  Its results must agree with the
regular workspace entry point's, within the tolerance the other tests use, on
two calls in a row (the shared array keeps the previous call's contents).
This file is collected last so that a failure here stops a run only after
every other test has run; it also passes when run on its own.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu

CASES = [(syn.Q4_0, 960, 960), (syn.Q4_0, 2048, 11008), (syn.Q4_0, 65, 1376),
         (syn.Q8_0, 5632, 2048), (syn.I8_B64, 100, 640), (syn.Q6_K, 4000, 2048)]


@pytest.mark.parametrize("fmt,N,K", CASES)
def test_fixed_workspace_matches_caller_workspace(fmt, N, K):
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    W, x = syn.make_problem(fmt, N, K, 1, seed=(40, fmt, N, K))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, 1)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y_ws = torch.empty((1, N), device="cuda")
    lean.lean_qmatmul_ws(fmt, Wd, xd, y_ws, N, K, 1, 0, ws, nb)
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=4)
    for _ in range(2):  # two calls in a row on the shared array
        y_fixed = torch.full((1, N), float("nan"), device="cuda")
        lean.lean_qmatmul_fixed_ws(fmt, Wd, xd, y_fixed, N, K)
        torch.cuda.synchronize()
        a = y_fixed.cpu().numpy().astype(np.float64)
        b = y_ws.cpu().numpy().astype(np.float64)
        check_close(a, b, bound, "fixed vs caller workspace")
        check_close(a, y_ref, bound, "fixed vs oracle")
    assert lean.lean_device_error(True) == 0


def test_fixed_workspace_limits():
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    assert lean.lean_fixed_workspace_bytes() == 3 << 20
    f = lean._lib.lean_qmatmul_fixed_ws
    buf = torch.zeros(64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # N beyond 262144 row groups is refused before any launch
    assert f(0, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), 262144 * 32 + 1, 32, 0,
             st) == lean.LEAN_ERR_SHAPE
    assert f(9, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), 32, 32, 0, st) == lean.LEAN_ERR_FORMAT
    assert f(0, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), 32, 48, 0, st) == lean.LEAN_ERR_SHAPE


@pytest.mark.parametrize("flags", [0, 1], ids=["plain", "early_weights"])
def test_fixed_workspace_in_captured_graph(flags):
    """The use the entry point exists for: after one warm call on the device,
    the call is recorded by stream capture (its counter clear and its kernel
    both become graph nodes), and the graph replayed twice into NaN-filled y
    gives the caller-workspace result and stays within the oracle's
    tolerance.  A call the library rejects inside the capture queues nothing
    and leaves the capture usable."""
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    fmt, N, K = syn.Q4_0, 2048, 11008
    W, x = syn.make_problem(fmt, N, K, 1, seed=(41, flags))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, 1)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y_ws = torch.empty((1, N), device="cuda")
    lean.lean_qmatmul_ws(fmt, Wd, xd, y_ws, N, K, 1, 0, ws, nb)
    y = torch.full((1, N), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lean.lean_qmatmul_fixed_ws(fmt, Wd, xd, y, N, K, flags, s)  # first call: set-up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            bad = lean._lib.lean_qmatmul_fixed_ws(fmt, Wd.data_ptr(), xd.data_ptr(), y.data_ptr(),
                                                  N, K + 1, flags, s.cuda_stream)
            lean.lean_qmatmul_fixed_ws(fmt, Wd, xd, y, N, K, flags, s)
    assert bad == lean.LEAN_ERR_SHAPE
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=4)
    for _ in range(2):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        a = y.cpu().numpy().astype(np.float64)
        check_close(a, y_ws.cpu().numpy().astype(np.float64), bound, "graph vs caller workspace")
        check_close(a, y_ref, bound, "graph vs oracle")
    assert lean.lean_device_error(True) == 0
