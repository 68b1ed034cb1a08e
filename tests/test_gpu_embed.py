"""GPU parity of lean_embed_rows, the embedding lookup: selected rows of a
quantized table as fp32, bit for bit the oracle's decoded weights.

The "lean" README keeps the embedding of its models as Q6_K (model table), and
the "oxinfer" crate page dequantizes a quantized table one row per token
(Pre-quantized checkpoints).  Covered: every format, ids in any order with
repeats, the first and last rows of the table and of a 32-row group, a single
id and many, the Qwen2.5-3B vocabulary (151936 x 2048, Q6_K) on sampled ids,
and an id out of range (its row NaN, the device error bit set, the others
right).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from lean_testlib import torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [syn.Q4_0, syn.Q8_0, syn.I8_B64, syn.Q6_K]
IDS = [syn.FORMAT_NAMES[f] for f in FMTS]


@pytest.fixture(scope="module")
def lean():
    torch_cuda()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def rows_ref(fmt, W, ids, K):
    """The oracle's exact weights of rows `ids` (canonical rows), as fp32."""
    sub = np.ascontiguousarray(W[np.asarray(ids)])
    return oracle.dequant(fmt, sub, len(ids), K).astype(np.float32)


def gather(lean, fmt, Wd, ids, N, K):
    torch = torch_cuda()
    idd = torch.tensor(np.asarray(ids, np.int32), device="cuda")
    out = torch.full((len(ids), K), float("inf"), device="cuda")
    lean.lean_embed_rows(fmt, Wd, idd, out, len(ids), N, K)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_embed_rows_bit_exact(lean, fmt):
    be = syn.BLOCK_ELEMS[fmt]
    N, K = 333, (8 if fmt == syn.Q6_K else 40) * be
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(80, fmt))
    Wd = lean.upload_packed(fmt, W, N, K)
    rng = np.random.default_rng((81, fmt))
    for ids in ([0], [N - 1], [31, 32, 33, 0, N - 1, 31],
                list(rng.integers(0, N, 200)), list(range(N))):
        got = gather(lean, fmt, Wd, ids, N, K)
        ref = rows_ref(fmt, W, ids, K)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (fmt, ids[:6])
    assert lean.lean_device_error(True) == 0


def test_embed_rows_qwen_vocabulary(lean):
    """The Qwen2.5-3B Q6_K table (151936 x 2048), sampled ids."""
    (lin,) = syn.qwen25_3b_lm_head().linears
    W, _ = lin.make()
    Wd = lean.upload_packed(lin.fmt, W, lin.N, lin.K)
    rng = np.random.default_rng(82)
    ids = [0, 1, 31, 32, lin.N - 33, lin.N - 1] + list(rng.integers(0, lin.N, 122))
    got = gather(lean, lin.fmt, Wd, ids, lin.N, lin.K)
    ref = rows_ref(lin.fmt, W, ids, lin.K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert lean.lean_device_error(True) == 0


@pytest.mark.parametrize("fmt", [syn.Q4_0, syn.Q6_K], ids=["q4_0", "q6_k"])
def test_embed_id_out_of_range(lean, fmt):
    be = syn.BLOCK_ELEMS[fmt]
    N, K = 70, 4 * be
    W, _ = syn.make_problem(fmt, N, K, 1, seed=(83, fmt))
    Wd = lean.upload_packed(fmt, W, N, K)
    assert lean.lean_device_error(True) == 0
    ids = [3, N, 5, -1, N - 1]
    got = gather(lean, fmt, Wd, ids, N, K)
    assert lean.lean_device_error(False) == 16
    assert lean.lean_device_error(True) == 16 and lean.lean_device_error(True) == 0
    assert np.isnan(got[1]).all() and np.isnan(got[3]).all()
    good = [0, 2, 4]
    ref = rows_ref(fmt, W, [ids[i] for i in good], K)
    assert np.array_equal(got[good].view(np.uint32), ref.view(np.uint32))


def test_embed_argument_errors(lean):
    torch = torch_cuda()
    W, _ = syn.make_problem(syn.Q6_K, 32, 256, 1, seed=(84,))
    Wd = lean.upload_packed(syn.Q6_K, W, 32, 256)
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.empty((4, 256), device="cuda")
    f = lean._lib.lean_embed_rows
    st = torch.cuda.current_stream().cuda_stream
    a = (Wd.data_ptr(), ids.data_ptr(), out.data_ptr())
    assert f(9, *a, 4, 32, 256, st) == lean.LEAN_ERR_FORMAT
    assert f(3, *a, 0, 32, 256, st) == lean.LEAN_ERR_SHAPE
    assert f(3, *a, 4, 32, 200, st) == lean.LEAN_ERR_SHAPE
    assert f(3, None, ids.data_ptr(), out.data_ptr(), 4, 32, 256, st) == lean.LEAN_ERR_NULL
    assert f(3, Wd.data_ptr(), ids.data_ptr(), out.data_ptr() + 4, 4, 32, 256, st) == lean.LEAN_ERR_ALIGN
    assert f(3, *a, 4, 32, 256, st) == lean.LEAN_OK
    torch.cuda.synchronize()
    assert lean.lean_device_error(True) == 0
