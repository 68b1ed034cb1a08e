"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bar: unpacked weights bit-exact; one-hot products bit-exact; every output
within |y - y_ref| <= 1e-4 * sum_k |w x| + 1e-6.
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


# ---- unpacked values: bit-exact ------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_dequant_bit_exact(lean, fmt):
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    for N, K in ((1, be), (33, 3 * be), (70, 11 * be), (64, 40 * be)):
        W, _ = syn.make_problem(fmt, N, K, 1, seed=(20, fmt, N, K))
        Wd = lean.upload_packed(fmt, W, N, K)
        wd = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
        lean.lean_dequant(fmt, Wd, wd, N, K)
        torch.cuda.synchronize()
        got = wd.cpu().numpy()
        ref = oracle.dequant(fmt, W, N, K).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (fmt, N, K)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_one_hot_bit_exact(lean, fmt):
    """x = e_k: y[n] must equal w[n,k] exactly (one nonzero product)."""
    be = syn.BLOCK_ELEMS[fmt]
    N, K = 37, 5 * be
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(21, fmt))
    ks = sorted(set([0, 1, 15, 16, 17, 31, be - 1, be, K // 2, K - 2, K - 1]))
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    w = oracle.dequant(fmt, W, N, K)
    for M in (1, len(ks)):
        y = run_gpu(fmt, W, x[:M], N, K)
        assert np.array_equal(y, w[:, ks[:M]].T), (fmt, M)


# ---- random problems: tolerance -------------------------------------------------

SHAPES = [(1, 1, 1), (32, 1, 1), (33, 2, 1), (100, 9, 1), (960, 30, 1), (65, 43, 1),
          (130, 7, 2), (50, 9, 3), (77, 12, 4), (64, 10, 7), (72, 11, 8), (48, 5, 9),
          (96, 17, 16), (40, 6, 17)]


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("N,nblk,M", SHAPES)
def test_parity_random(lean, fmt, N, nblk, M):
    be = syn.BLOCK_ELEMS[fmt]
    if fmt == syn.Q6_K:
        nblk = max(1, nblk // 4)
    K = nblk * be
    W, x = syn.make_problem(fmt, N, K, M, seed=(22, fmt, N, K, M))
    y = run_gpu(fmt, W, x, N, K)
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K, threads=4)
    check_close(y, y_ref, bound, "%s N=%d K=%d M=%d" % (syn.FORMAT_NAMES[fmt], N, K, M))


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_deterministic_and_canary(lean, fmt):
    """Same inputs -> same bits; nothing written outside y."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    N, K, M = 70, 8 * be, 3
    W, x = syn.make_problem(fmt, N, K, M, seed=(23, fmt))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    buf = torch.full((M * N + 64,), float("nan"), dtype=torch.float32, device="cuda")
    lean.lean_qmatmul(fmt, Wd, xd, buf, N, K, M)
    a = buf.clone()
    lean.lean_qmatmul(fmt, Wd, xd, buf, N, K, M)
    torch.cuda.synchronize()
    assert torch.equal(a[:M * N].view(torch.int32), buf[:M * N].view(torch.int32))
    assert torch.isnan(buf[M * N:]).all()
    assert not torch.isnan(buf[:M * N]).any()


# ---- argument errors are returned before any launch ----------------------------

def test_argument_errors(lean):
    torch = torch_cuda()
    N, K = 32, 64
    W, x = syn.make_problem(syn.Q4_0, N, K, 1, seed=(24,))
    Wd = lean.upload_packed(syn.Q4_0, W, N, K)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty((1, N), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    f = lean._lib.lean_qmatmul
    assert f(7, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 1, st) == lean.LEAN_ERR_FORMAT
    assert f(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, 48, 1, st) == lean.LEAN_ERR_SHAPE
    assert f(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), 0, K, 1, st) == lean.LEAN_ERR_SHAPE
    assert f(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 0, st) == lean.LEAN_ERR_SHAPE
    assert f(0, None, xd.data_ptr(), yd.data_ptr(), N, K, 1, st) == lean.LEAN_ERR_NULL
    assert f(0, Wd.data_ptr(), xd.data_ptr() + 4, yd.data_ptr(), N, K, 1, st) == lean.LEAN_ERR_ALIGN
    assert f(0, Wd.data_ptr() + 8, xd.data_ptr(), yd.data_ptr(), N, K, 1, st) == lean.LEAN_ERR_ALIGN
    # a good call still works afterwards
    assert f(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 1, st) == lean.LEAN_OK
    torch.cuda.synchronize()


def test_streams_and_graph_capture(lean):
    """Calls run on the given stream and can be captured into a CUDA graph."""
    torch = torch_cuda()
    fmt, N, K = syn.Q4_0, 256, 512
    W, x = syn.make_problem(fmt, N, K, 1, seed=(25,))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    yd = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        lean.lean_qmatmul(fmt, Wd, xd, yd, N, K, 1, s)  # warm-up outside capture
        s.synchronize()
        yd.zero_()
        with torch.cuda.graph(g, stream=s):
            lean.lean_qmatmul(fmt, Wd, xd, yd, N, K, 1, s)
    g.replay()
    torch.cuda.synchronize()
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
    check_close(yd.cpu().numpy().astype(np.float64), y_ref, bound, "graph replay")


@pytest.mark.parametrize("M,extra", [(1, 0), (1, 4), (3, 0)], ids=["m1_one_wave", "m1_stream", "m3"])
def test_early_weights_chain_orders_x(lean, M, extra):
    """A chain y_{i+1} = W_i y_i with programmatic dependent launch: each
    product must read its x only after the previous one wrote it.  The chain is
    run with and without the flag (and inside a CUDA graph); results must match
    bit for bit, and the buffers start as NaN so a premature read shows.  M = 1
    on the one-wave kernel and (LEAN_FLAG_STREAM) on the streaming kernel."""
    torch = torch_cuda()
    fmt, N = syn.Q4_0, 960
    steps = 24
    Ws = []
    for i in range(steps):
        W, _ = syn.make_problem(fmt, N, N, 1, seed=(26, i))
        Ws.append(lean.upload_packed(fmt, W, N, N))
    _, x0 = syn.make_problem(fmt, N, N, M, seed=(27,))
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
        ref = chain(extra, s)
        pdl = chain(lean.LEAN_FLAG_EARLY_WEIGHTS | extra, s)
    s.synchronize()
    for a, b in zip(ref, pdl):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.isfinite(ref[-1]).all()
    # the same chain captured into a graph
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        bufs = [torch.full((M, N), float("nan"), device="cuda") for _ in range(steps)]
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            cur = x0d
            for i in range(steps):
                lean.lean_qmatmul_ex(fmt, Ws[i], cur, bufs[i], N, N, M,
                                     lean.LEAN_FLAG_EARLY_WEIGHTS | extra, s)
                cur = bufs[i]
    for _ in range(3):
        for b in bufs:
            b.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, bufs):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_flags_rejected(lean):
    torch = torch_cuda()
    N, K = 32, 64
    W, x = syn.make_problem(syn.Q4_0, N, K, 1, seed=(28,))
    Wd = lean.upload_packed(syn.Q4_0, W, N, K)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty((1, N), device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lean._lib.lean_qmatmul_ex(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 1, 16,
                                     st) == lean.LEAN_ERR_FORMAT
    # the streaming-kernel flag is known
    assert lean._lib.lean_qmatmul_ex(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 1,
                                     lean.LEAN_FLAG_STREAM, st) == lean.LEAN_OK
    # the x-planes flag is known (and ignored without a workspace)
    assert lean._lib.lean_qmatmul_ex(0, Wd.data_ptr(), xd.data_ptr(), yd.data_ptr(), N, K, 1,
                                     lean.LEAN_FLAG_X_PLANES, st) == lean.LEAN_OK
    torch.cuda.synchronize()


# ---- workspace (stream-K split of row groups) and batched launches -------------

WS_SHAPES = [(1, 1), (33, 3), (64, 43), (100, 17), (32, 200), (65, 9)]


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("N,nblk", WS_SHAPES)
@pytest.mark.parametrize("flags", [0, 2, 4], ids=["one_wave", "x_planes", "stream_fp32_x"])
def test_workspace_split_groups(lean, fmt, N, nblk, flags):
    """M = 1 with a workspace: on the streaming kernel (LEAN_FLAG_STREAM, or x
    as integer planes: dp4a, Q6_K ignores that flag) row groups split between
    CTAs are completed by the last CTA; two calls in a row (the counters must
    come back zeroed); without either flag these shapes take the one-wave
    kernel, which leaves the workspace alone."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    if fmt == syn.Q6_K:
        nblk = max(1, nblk // 3)
    K = nblk * be
    W, x = syn.make_problem(fmt, N, K, 1, seed=(29, fmt, N, K))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    nb = lean.lean_qmatmul_workspace_bytes(fmt, N, K, 1)
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
    outs = []
    for _ in range(2):
        yd = torch.full((1, N), float("nan"), device="cuda")
        lean.lean_qmatmul_ws(fmt, Wd, xd, yd, N, K, 1, flags, ws, nb)
        torch.cuda.synchronize()
        y = yd.cpu().numpy().astype(np.float64)
        check_close(y, y_ref, bound, "ws %s N=%d K=%d" % (syn.FORMAT_NAMES[fmt], N, K))
        outs.append(y)
    assert np.array_equal(outs[0], outs[1])
    # the arrival counters (the workspace's last 256-byte-rounded 4 * groups
    # bytes) must be back to zero; the rest is scratch
    cnt_bytes = (4 * ((N + 31) // 32) + 255) // 256 * 256
    assert int(ws[nb - cnt_bytes:].count_nonzero()) == 0
    assert lean.lean_device_error(True) == 0


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("use_ws", [0, 1, 2, 3, 4],
                         ids=["one_wave", "one_wave_ws", "x_planes", "stream_whole_groups",
                              "stream_workspace"])
def test_batch(lean, fmt, use_ws):
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    shapes = [(1, 1), (40, 3), (960, 30), (33, 8), (320, 17), (64, 1), (100, 9)]
    if fmt == syn.Q6_K:
        shapes = [(N, max(1, n // 4)) for N, n in shapes]
    items, keep, refs = [], [], []
    for i, (N, nblk) in enumerate(shapes):
        K = nblk * be
        W, x = syn.make_problem(fmt, N, K, 1, seed=(30, fmt, i))
        Wd = lean.upload_packed(fmt, W, N, K)
        xd = torch.from_numpy(x).cuda()
        yd = torch.full((N,), float("nan"), device="cuda")
        keep += [Wd, xd, yd]
        items.append((Wd, xd, yd, N, K))
        refs.append(oracle.qmatmul(fmt, W, x, N, K))
    probs = lean.make_problems(items)
    ws, nb = None, 0
    if use_ws in (1, 2, 4):
        nb = lean.lean_batch_workspace_bytes(fmt, probs)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for it in items:
            it[2].fill_(float("nan"))
        flags = lean.LEAN_FLAG_EARLY_WEIGHTS | (lean.LEAN_FLAG_X_PLANES if use_ws == 2 else 0) | \
            (lean.LEAN_FLAG_STREAM if use_ws >= 3 else 0)
        lean.lean_qmatmul_batch(fmt, probs, flags, ws, nb)
        torch.cuda.synchronize()
        for (Wd, xd, yd, N, K), (y_ref, bound) in zip(items, refs):
            check_close(yd.cpu().numpy().astype(np.float64)[None, :], y_ref, bound,
                        "batch N=%d K=%d" % (N, K))
    assert lean.lean_device_error(True) == 0


def test_batch_argument_errors(lean):
    torch = torch_cuda()
    W, x = syn.make_problem(syn.Q4_0, 32, 64, 1, seed=(31,))
    Wd = lean.upload_packed(syn.Q4_0, W, 32, 64)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty(32, device="cuda")
    good = lean.make_problems([(Wd, xd, yd, 32, 64)])
    f = lean._lib.lean_qmatmul_batch
    st = torch.cuda.current_stream().cuda_stream
    import ctypes
    p = ctypes.cast(good, ctypes.c_void_p)
    assert f(0, 0, p, 0, None, 0, st) == lean.LEAN_ERR_SHAPE
    assert f(0, 257, p, 0, None, 0, st) == lean.LEAN_ERR_SHAPE
    assert f(0, 1, None, 0, None, 0, st) == lean.LEAN_ERR_NULL
    assert f(9, 1, p, 0, None, 0, st) == lean.LEAN_ERR_FORMAT
    bad = lean.make_problems([(Wd, xd, yd, 32, 48)])
    assert f(0, 1, ctypes.cast(bad, ctypes.c_void_p), 0, None, 0, st) == lean.LEAN_ERR_SHAPE
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    assert f(0, 1, p, 0, ws.data_ptr(), 64, st) == lean.LEAN_ERR_SHAPE  # too small
    assert f(0, 1, p, 0, None, 0, st) == lean.LEAN_OK
    torch.cuda.synchronize()


def test_bounded_wait_times_out(lean):
    """A bounded wait on a barrier that nothing completes gives up, sets its bit
    of the device error word and leaves the context usable."""
    import time
    torch = torch_cuda()
    assert lean.lean_device_error(True) == 0
    assert lean._lib.lean_wait_selftest(0, None) == lean.LEAN_ERR_SHAPE
    assert lean._lib.lean_wait_selftest(1000001, None) == lean.LEAN_ERR_SHAPE
    t0 = time.perf_counter()
    lean.lean_wait_selftest(20000)  # 20 ms
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert 0.015 < took < 2.0, took
    assert lean.lean_device_error(False) == 8
    assert lean.lean_device_error(True) == 8
    assert lean.lean_device_error(True) == 0
    # the context still runs products
    fmt, N, K = syn.Q4_0, 96, 256
    W, x = syn.make_problem(fmt, N, K, 1, seed=(32,))
    Wd = lean.upload_packed(fmt, W, N, K)
    xd = torch.from_numpy(x).cuda()
    yd = torch.full((1, N), float("nan"), device="cuda")
    lean.lean_qmatmul(fmt, Wd, xd, yd, N, K, 1)
    torch.cuda.synchronize()
    y_ref, bound = oracle.qmatmul(fmt, W, x, N, K)
    check_close(yd.cpu().numpy().astype(np.float64), y_ref, bound, "after self-test")
    assert lean.lean_device_error(True) == 0


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("planes", [0, 1], ids=["fp32_x", "x_planes"])
def test_batch_run_time_handout(lean, fmt, planes):
    """A batch with at least three group blocks (256 rows) per CTA slot takes
    whole group blocks at run time, largest first: every row is right, two
    calls on one workspace agree bit for bit, and the counters end at zero."""
    torch = torch_cuda()
    be = syn.BLOCK_ELEMS[fmt]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nprob = 256
    per = -(-3 * 2 * sms // nprob) + 1  # group blocks per problem
    items, keep, refs, groups = [], [], [], 0
    for i in range(nprob):
        N = 256 * per - (0 if i % 3 else 200)  # some problems end in a partial block
        K = be * (1 + i % 4) * (1 if fmt == syn.Q6_K else 2)
        W, x = syn.make_problem(fmt, N, K, 1, seed=(33, fmt, i))
        Wd = lean.upload_packed(fmt, W, N, K)
        xd = torch.from_numpy(x).cuda()
        yd = torch.full((N,), float("nan"), device="cuda")
        keep += [Wd, xd, yd]
        items.append((Wd, xd, yd, N, K))
        refs.append(oracle.qmatmul(fmt, W, x, N, K))
        groups += (N + 31) // 32
    probs = lean.make_problems(items)
    nb = lean.lean_batch_workspace_bytes(fmt, probs)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    flags = lean.LEAN_FLAG_EARLY_WEIGHTS | (lean.LEAN_FLAG_X_PLANES if planes else 0)
    outs = []
    for rep in range(2):
        for it in items:
            it[2].fill_(float("nan"))
        lean.lean_qmatmul_batch(fmt, probs, flags, ws, nb)
        torch.cuda.synchronize()
        ys = []
        for (Wd, xd, yd, N, K), (y_ref, bound) in zip(items, refs):
            y = yd.cpu().numpy().astype(np.float64)[None, :]
            check_close(y, y_ref, bound, "handout N=%d K=%d" % (N, K))
            ys.append(y)
        outs.append(np.concatenate(ys, axis=1))
    assert np.array_equal(outs[0], outs[1])
    # arrival counters and the two hand-out counters: the workspace's tail
    cnt_bytes = (4 * (groups + 2) + 255) // 256 * 256
    assert int(ws[nb - cnt_bytes:].count_nonzero()) == 0
    assert lean.lean_device_error(True) == 0
