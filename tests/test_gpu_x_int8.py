"""GPU parity of the int8-activation variant (LEAN_FLAG_X_INT8): x quantized
to int8 per 32 elements, int8 dot products ("oxinfer" crate page, How it
works: per-matmul activation quantization ahead of int8 SDOT).

Against the oracle that quantizes x by the same rule (oracle.qmatmul_x_int8):
  - the codes and scales bit for bit, through rows holding one weight of 1
    (then y[n] = s * q[n], one fp32 rounding of an exact value on both sides);
  - random problems, single calls and batches (up to a whole decode step),
    within |y - y~| <= 1e-4 * sum|w x~| + 1e-6, x~ the dequantized activations;
  - outlier channels (the rule is what it is: their blocks lose the small
    values, on both sides alike);
  - argument errors (Q6_K, no workspace, M != 1, the fixed-workspace entry).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def run_int8(lean, fmt, items, batch):
    """items: [(W canonical, x, N, K)]; returns the list of y (fp64)."""
    torch = torch_cuda()
    dev = []
    for W, x, N, K in items:
        Wd = lean.upload_packed(fmt, W, N, K)
        xd = torch.from_numpy(np.ascontiguousarray(x, np.float32).reshape(-1)).cuda()
        yd = torch.full((N,), float("nan"), device="cuda")
        dev.append((Wd, xd, yd, N, K))
    flags = lean.LEAN_FLAG_X_INT8 | lean.LEAN_FLAG_EARLY_WEIGHTS
    if batch:
        probs = lean.make_problems(dev)
        nb = lean.lean_batch_workspace_bytes(fmt, probs)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
        lean.lean_qmatmul_batch(fmt, probs, flags, ws, nb)
    else:
        for Wd, xd, yd, N, K in dev:
            nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, 1)
            ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
            lean.lean_qmatmul_ws(fmt, Wd, xd, yd, N, K, 1, flags, ws, nb)
    torch.cuda.synchronize()
    assert lean.lean_device_error(True) == 0
    return [d[2].cpu().numpy().astype(np.float64)[None, :] for d in dev]


def unit_rows(fmt, K):
    """Canonical N = K rows, row n holding weight 1 at column n and 0 elsewhere."""
    be, bb = syn.BLOCK_ELEMS[fmt], syn.BLOCK_BYTES[fmt]
    W = np.zeros((K, K // be, bb), np.uint8)
    one = np.array([1.0], np.float16).view(np.uint8)
    W[:, :, 0:2] = one
    if fmt == syn.Q4_0:
        W[:, :, 2:] = 0x88  # q = 8 everywhere: weight 0
    for n in range(K):
        b, j = divmod(n, be)
        if fmt == syn.Q4_0:
            if j < 16:
                W[n, b, 2 + j] = (W[n, b, 2 + j] & 0xF0) | 9
            else:
                W[n, b, 2 + j - 16] = (W[n, b, 2 + j - 16] & 0x0F) | 0x90
        else:
            W[n, b, 2 + j] = 1
    return W.reshape(K, -1)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_codes_and_scales_bit_exact(lean, fmt):
    K = 512
    W = unit_rows(fmt, K)
    rng = np.random.default_rng((110, fmt))
    x = (rng.standard_normal(K) * np.exp(rng.uniform(-4, 4, K // 32)).repeat(32)).astype(np.float32)
    x[[0, 33, 100]] = [0.0, 5e3, -7e-3]
    x[64:96] = 0.0  # a zero block
    (y,) = run_int8(lean, fmt, [(W, x, K, K)], batch=False)
    y_ref, _ = oracle.qmatmul_x_int8(fmt, W, x, K, K)  # = s * q, exact in fp64
    assert np.array_equal(y.astype(np.float32), y_ref.astype(np.float32))
    xq, sc = oracle.quantize_x_int8(x[None, :])
    assert np.array_equal(y_ref[0], np.repeat(sc[0].astype(np.float64), 32) * xq[0])


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("batch", [False, True], ids=["single", "batch"])
def test_random_problems(lean, fmt, batch):
    be = syn.BLOCK_ELEMS[fmt]
    shapes = [(1, 2 * be), (33, 3 * be), (300, 32 * be), (960, 960 // be * be or be), (65, 43 * be)]
    items = []
    for i, (N, K) in enumerate(shapes):
        K = max(be, K // be * be)
        W, x = syn.make_problem(fmt, N, K, 1, seed=(111, fmt, i))
        items.append((W, x, N, K))
    ys = run_int8(lean, fmt, items, batch)
    for (W, x, N, K), y in zip(items, ys):
        y_ref, bound = oracle.qmatmul_x_int8(fmt, W, x, N, K)
        check_close(y, y_ref, bound, "x int8 %s N=%d K=%d" % (syn.FORMAT_NAMES[fmt], N, K))
        # a different product from the fp32-x one
        y32, b32 = oracle.qmatmul(fmt, W, x, N, K)
        if N * K > 10000:
            assert np.mean(np.abs(y - y32) > 1e-4 * b32 + 1e-6) > 0.3


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_outlier_channels(lean, fmt):
    rng = np.random.default_rng((112, fmt))
    N, K = 200, 2048
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(113, fmt))
    x = rng.standard_normal(K).astype(np.float32)
    x[np.arange(5, K, 96)] = 2e4
    (y,) = run_int8(lean, fmt, [(W, x, N, K)], batch=False)
    y_ref, bound = oracle.qmatmul_x_int8(fmt, W, x, N, K)
    check_close(y, y_ref, bound, "outliers")


def test_decode_step_batch(lean):
    """The 224 linears of the SmolLM2-360M step in one call, sampled linears
    against the oracle."""
    lins = syn.smollm2_360m_decode_stack().linears
    items = [lin.make() + (lin.N, lin.K) for lin in lins]
    ys = run_int8(lean, syn.Q4_0, items, batch=True)
    for i in (0, 1, 3, 4, 6, 100, 223):
        W, x, N, K = items[i]
        y_ref, bound = oracle.qmatmul_x_int8(syn.Q4_0, W, x, N, K)
        check_close(ys[i], y_ref, bound, lins[i].name)


def test_argument_errors(lean):
    torch = torch_cuda()
    W, x = syn.make_problem(syn.Q4_0, 64, 256, 2, seed=(114,))
    Wd = lean.upload_packed(syn.Q4_0, W, 64, 256)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty((2, 64), device="cuda")
    nb = lean.lean_qmatmul_workspace_bytes(0, 64, 256, 1)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    f = lean._lib.lean_qmatmul_ws
    st = torch.cuda.current_stream().cuda_stream
    F = lean.LEAN_FLAG_X_INT8
    a = (Wd.data_ptr(), xd.data_ptr(), yd.data_ptr())
    assert f(0, *a, 64, 256, 1, F, None, 0, st) == lean.LEAN_ERR_NULL
    assert f(0, *a, 64, 256, 2, F, ws.data_ptr(), nb, st) == lean.LEAN_ERR_FORMAT
    W6, _ = syn.make_problem(syn.Q6_K, 64, 256, 1, seed=(115,))
    W6d = lean.upload_packed(syn.Q6_K, W6, 64, 256)
    assert f(3, W6d.data_ptr(), xd.data_ptr(), yd.data_ptr(), 64, 256, 1, F, ws.data_ptr(), nb,
             st) == lean.LEAN_ERR_FORMAT
    assert lean._lib.lean_qmatmul_fixed_ws(0, *a, 64, 256, F, st) == lean.LEAN_ERR_FORMAT
    assert f(0, *a, 64, 256, 1, F, ws.data_ptr(), nb, st) == lean.LEAN_OK
    torch.cuda.synchronize()
