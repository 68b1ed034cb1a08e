"""Shared helpers for the GPU parity tests: upload, run through the C ABI,
compare with the oracle under |y - y_ref| <= 1e-4 * sum|w x| + 1e-6."""
import numpy as np

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn

REL_TOL = 1e-4
ABS_TOL = 1e-6


def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU test run without a GPU"
    return torch


def run_gpu(fmt, W_canon, x, N, K, stream=None, workspace=False):
    """Pack on the host, upload, call lean_qmatmul (or lean_qmatmul_ws with a
    workspace of the queried size), return y as float64 numpy."""
    torch = torch_cuda()
    from block_quantized_weight_dot_gb300 import lean
    Wd = lean.upload_packed(fmt, W_canon, N, K)
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)).cuda()
    M = xd.shape[0]
    yd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    if workspace:
        nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, M)
        ws = torch.zeros((max(nb, 256),), dtype=torch.uint8, device="cuda")
        lean.lean_qmatmul_ws(fmt, Wd, xd, yd, N, K, M, 0, ws, nb, stream)
    else:
        lean.lean_qmatmul(fmt, Wd, xd, yd, N, K, M, stream)
    torch.cuda.synchronize()
    return yd.cpu().numpy().astype(np.float64)


def check_close(y, y_ref, bound, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    lim = REL_TOL * bound + ABS_TOL
    bad = ~(err <= lim)  # NaN counts as bad
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d outputs out of tolerance; first at %s: y=%r ref=%r "
                             "bound=%r err=%r" % (what, int(bad.sum()), bad.size, tuple(i),
                                                  y[tuple(i)], y_ref[tuple(i)], bound[tuple(i)],
                                                  err[tuple(i)]))
    return float(np.max(err / lim)) if err.size else 0.0
