"""GPU parity of the tensor-core products (from lean_tensor_core_min_m(fmt)
rows of x: 9, Q6_K 5) against the fp64 oracle: up to 64 rows, integer codes times split-bf16 x with the block
scales applied per group after the MMAs; more rows, split-bf16 weights times
split-bf16 x in 256-row tiles of x.

Covers ragged row tiles (N not a multiple of 128), K tails (K not a multiple
of 64), K split over a thread-block cluster (few row tiles, long K), x tiles
with a ragged last one (both kernels), the switch-over from the CUDA-core
path (both sides of it, and 15 / 16 rows), bit-exact one-hot products for Q4_0 (exact in both),
determinism, writes confined to y, and the device error word left clear --
each both with a caller workspace (x split once by its own kernel) and
without one (each CTA splits its x).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import check_close, run_gpu, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64, syn.Q6_K]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


# (N, K in units of 256 elements, M); K is then trimmed per format below to
# reach tails that are not multiples of 64
SHAPES = [
    (128, 2, 32),     # one tile, switch-over size
    (130, 3, 33),     # ragged row tile, odd M
    (1000, 4, 64),    # several tiles
    (96, 32, 48),     # one tile, long K: K split over a cluster
    (96, 32, 20),     # the same with the epilogue's warp sets on alternate groups
    (160, 24, 9),     # the fewest rows of the tensor-core path, K split
    (300, 8, 256),    # a full 256-row tile of x
    (200, 2, 257),    # two tiles of x, the last with one row
    (64, 3, 300),     # rows of x ragged in the second tile
    (1, 4, 40),       # a single weight row
]


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("N,k256,M", SHAPES)
def test_mma_parity(lean, fmt, N, k256, M):
    be = syn.BLOCK_ELEMS[fmt]
    K = 256 * k256
    if be <= 64:
        K -= be  # leaves a K tail of 32 (Q4_0, Q8_0) or a full block (I8_B64)
    W, x = syn.make_problem(fmt, N, K, M, seed=(40, fmt, N, K, M))
    y = run_gpu(fmt, W, x, N, K)
    y_ws = run_gpu(fmt, W, x, N, K, workspace=True)  # x split once, by its own kernel
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=8)
    what = "%s N=%d K=%d M=%d" % (syn.FORMAT_NAMES[fmt], N, K, M)
    check_close(y, y_ref, bound, what)
    check_close(y_ws, y_ref, bound, what + " (workspace)")
    assert np.array_equal(y, y_ws)
    assert lean.lean_device_error(0) == 0


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_switch_over_agrees(lean, fmt):
    """Both sides of the switch from CUDA cores to tensor cores meet the bar,
    and so do 15 and 16 rows (one padded x tile on the tensor cores)."""
    m0 = lean.lean_tensor_core_min_m(fmt)
    assert m0 == (5 if fmt == syn.Q6_K else 9)
    N, K = 384, 2048
    for M in sorted({m0 - 1, m0, 15, 16}):
        W, x = syn.make_problem(fmt, N, K, M, seed=(41, fmt, M))
        y = run_gpu(fmt, W, x, N, K)
        y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=8)
        check_close(y, y_ref, bound, "%s M=%d" % (syn.FORMAT_NAMES[fmt], M))


def test_mma_one_hot_bit_exact_q4_0(lean):
    """Q4_0 weights split exactly into bf16 hi + lo, so x = e_k returns
    w[n, k] bit for bit through the tensor cores too."""
    fmt, N = syn.Q4_0, 200
    K = 32 * 13
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(42,))
    ks = list(range(0, K, 11))[:40]
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    w = oracle.dequant(fmt, W, N, K)
    y = run_gpu(fmt, W, x, N, K)
    assert np.array_equal(y, w[:, ks].T)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_mma_deterministic_and_canary(lean, fmt):
    """Same inputs give the same bits (the cluster sums run in rank order),
    and nothing is written outside y."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 160, 40 * be if be < 256 else 8 * be, 70
    W, x = syn.make_problem(fmt, N, K, M, seed=(43, fmt))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    buf = torch.full((M * N + 64,), float("nan"), dtype=torch.float32, device="cuda")
    lean.lean_qmatmul(fmt, Wd, xd, buf, N, K, M)
    a = buf.clone()
    lean.lean_qmatmul(fmt, Wd, xd, buf, N, K, M)
    torch.cuda.synchronize()
    assert torch.equal(a[:M * N].view(torch.int32), buf[:M * N].view(torch.int32))
    assert torch.isnan(buf[M * N:]).all()
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=8)
    check_close(buf[:M * N].cpu().numpy().astype(np.float64).reshape(M, N), y_ref, bound,
                "canary")


def test_mma_early_weights_chain(lean):
    """A chain y_{i+1} = W_i y_i of 48-row products with programmatic
    dependent launch, plain, and captured into a graph: identical bits."""
    torch = torch_cuda()
    fmt, N, M, steps = syn.Q4_0, 960, 48, 12
    Ws = []
    for i in range(steps):
        W, _ = syn.make_problem(fmt, N, N, 1, seed=(44, i))
        Ws.append(lean.upload_packed(fmt, W, N, N))
    _, x0 = syn.make_problem(fmt, N, N, M, seed=(45,))
    x0d = torch.from_numpy(x0 / np.float32(30.0)).cuda()

    def chain(flags, stream):
        bufs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(steps)]
        torch.cuda.synchronize()
        cur = x0d
        for i in range(steps):
            lean.lean_qmatmul_ex(fmt, Ws[i], cur, bufs[i], N, N, M, flags, stream)
            cur = bufs[i]
        return bufs

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ref = chain(0, s)
        pdl = chain(lean.LEAN_FLAG_EARLY_WEIGHTS, s)
    s.synchronize()
    for a, b in zip(ref, pdl):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.isfinite(ref[-1]).all()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        bufs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(steps)]
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            cur = x0d
            for i in range(steps):
                lean.lean_qmatmul_ex(fmt, Ws[i], cur, bufs[i], N, N, M,
                                     lean.LEAN_FLAG_EARLY_WEIGHTS, s)
                cur = bufs[i]
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, bufs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert lean.lean_device_error(0) == 0


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_mma_caller_workspace(lean, fmt):
    """With a caller-owned workspace (which then holds the split x, written
    once by its own kernel) the bits equal those of a call without one (where
    every CTA splits its own x; the library allocates nothing); a workspace
    smaller than the query says is refused before any launch."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 300, (4 if fmt == syn.Q6_K else 40) * be, 100
    W, x = syn.make_problem(fmt, N, K, M, seed=(46, fmt))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, M)
    assert nb >= M * K * 4
    ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device="cuda")  # contents do not matter
    y1 = torch.full((M, N), float("nan"), device="cuda")
    y2 = torch.full((M, N), float("nan"), device="cuda")
    lean.lean_qmatmul_ws(fmt, Wd, xd, y1, N, K, M, 0, ws, nb)
    lean.lean_qmatmul(fmt, Wd, xd, y2, N, K, M)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    with pytest.raises(lean.LeanError) as e:
        lean.lean_qmatmul_ws(fmt, Wd, xd, y1, N, K, M, 0, ws, nb - 16)
    assert e.value.status == lean.LEAN_ERR_SHAPE
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=8)
    check_close(y1.cpu().numpy().astype(np.float64), y_ref, bound, "caller workspace")
