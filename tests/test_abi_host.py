"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every function include/lean_qmatmul.h declares, and its host calls (sizes,
packing) behave as documented."""
import ctypes
import os
import re

import numpy as np
import pytest

from block_quantized_weight_dot_gb300 import build as lib_build
from block_quantized_weight_dot_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lean():
    lib_build.build()
    from block_quantized_weight_dot_gb300 import lean as L
    return L


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(lean_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_exports_every_declared_symbol(lean):
    names = declared_functions()
    assert "lean_qmatmul" in names and "lean_pack" in names
    lib = ctypes.CDLL(lean.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lean.SIGNATURES), "binding and header disagree"


def test_sizes(lean):
    for fmt in range(4):
        assert lean.lean_block_elems(fmt) == syn.BLOCK_ELEMS[fmt]
        assert lean.lean_block_bytes(fmt) == syn.BLOCK_BYTES[fmt]
        be = syn.BLOCK_ELEMS[fmt]
        assert lean.lean_canonical_bytes(fmt, 7, 3 * be) == syn.canonical_bytes(fmt, 7, 3 * be)
        assert lean.lean_packed_bytes(fmt, 7, 3 * be) >= syn.canonical_bytes(fmt, 7, 3 * be)
        assert lean.lean_packed_bytes(fmt, 7, be + 1) == -1
        assert lean.lean_packed_bytes(fmt, 0, be) == -1
    assert lean.lean_block_elems(9) == 0
    # Q4_0 960x960: 30 groups x 30 vectors x 512 B + 30 groups x 4 scale vectors x 512 B
    assert lean.lean_packed_bytes(0, 960, 960) == 30 * 30 * 512 + 30 * 4 * 512


def test_workspace_sizes(lean):
    """M = 1: stream-K scratch; fewer rows than the tensor-core switch (9,
    Q6_K 5): none; from it on: x split into bf16 hi + lo (4 bytes per element)
    over rows padded to 16 within each 256-row tile and K padded to 64."""
    assert lean.lean_qmatmul_workspace_bytes(0, 960, 960, 1) > 0
    assert [lean.lean_tensor_core_min_m(f) for f in range(4)] == [9, 9, 9, 5]
    assert lean.lean_tensor_core_min_m(7) == -1
    assert lean.lean_qmatmul_workspace_bytes(0, 960, 960, 8) == 0
    assert lean.lean_qmatmul_workspace_bytes(0, 960, 960, 9) == 16 * 960 * 4
    assert lean.lean_qmatmul_workspace_bytes(3, 960, 1024, 4) == 0
    assert lean.lean_qmatmul_workspace_bytes(3, 960, 1024, 5) == 16 * 1024 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 960, 960, 16) == 16 * 960 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 2048, 2048, 256) == 256 * 2048 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 2048, 2048, 32) == 32 * 2048 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 100, 96, 33) == 48 * 128 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 100, 96, 257) == (256 + 16) * 128 * 4
    assert lean.lean_qmatmul_workspace_bytes(0, 100, 96, 0) == -1


def test_m1_workspace_layout(lean):
    """M = 1 workspace: 2 MiB of stream-K partial sums (512 CTAs x 2 sides x
    16 groups x 32 rows, fp32), then x as planes (160 bytes per 32 elements,
    integer formats), then one counter per 32-row group, plus the two counters
    of the run-time hand-out for a batch of two or more; each region rounded up
    to 256 bytes."""
    part = 512 * 2 * 16 * 32 * 4
    r = lambda b: (b + 255) // 256 * 256
    assert lean.lean_qmatmul_workspace_bytes(0, 960, 960, 1) == part + r(30 * 160) + r(30 * 4)
    assert lean.lean_qmatmul_workspace_bytes(3, 1000, 512, 1) == part + r(32 * 4)  # Q6_K: fp32 x
    two = lean.make_problems([(None, None, None, 960, 960), (None, None, None, 320, 2560)])
    assert lean.lean_batch_workspace_bytes(0, two) == part + r((30 + 80) * 160) + r((30 + 10 + 2) * 4)
    one = lean.make_problems([(None, None, None, 960, 960)])
    assert lean.lean_batch_workspace_bytes(0, one) == lean.lean_qmatmul_workspace_bytes(0, 960, 960, 1)
    bad = lean.make_problems([(None, None, None, 960, 961)])
    assert lean.lean_batch_workspace_bytes(0, bad) == -1


@pytest.mark.parametrize("fmt", range(4), ids=[syn.FORMAT_NAMES[f] for f in range(4)])
def test_pack_round_trip(lean, fmt):
    be = syn.BLOCK_ELEMS[fmt]
    for N, K in ((1, be), (33, 3 * be), (70, 11 * be), (31, 17 * be)):
        W, _ = syn.make_problem(fmt, N, K, 1, seed=(1, fmt, N))
        p = lean.lean_pack(fmt, W, N, K)
        assert lean.lean_unpack_canonical(fmt, p, N, K).tobytes() == W.tobytes()
    # edge blocks: all-zero, all-ones bytes
    for fill in (0x00, 0xFF, 0x80, 0x7F):
        W = np.full(syn.canonical_bytes(fmt, 3, 2 * be), fill, np.uint8)
        p = lean.lean_pack(fmt, W, 3, 2 * be)
        assert lean.lean_unpack_canonical(fmt, p, 3, 2 * be).tobytes() == W.tobytes()


def test_pack_padding_is_zero(lean):
    """Rows past N in the last 32-row group and unused scale slots are zeros."""
    fmt, N, K = 0, 33, 64  # two blocks: one step of 2 quant vectors + 1 scale vector
    W = np.full(syn.canonical_bytes(fmt, N, K), 0xFF, np.uint8)
    p = lean.lean_pack(fmt, W, N, K).reshape(2, 3, 32, 16)  # [group][vector][row][16 B]
    assert (p[0, :2] == 0xFF).all()                 # group 0: every row present
    assert (p[1, :, 1:, :] == 0).all()              # group 1: rows 33..63 are padding
    assert (p[1, :2, 0, :] == 0xFF).all()           # row 32's quant vectors
    assert (p[1, 2, 0, :4] == 0xFF).all() and (p[1, 2, 0, 4:] == 0).all()  # 2 of 8 scales


def test_host_argument_errors(lean):
    f = lean._lib.lean_pack
    buf = np.zeros(1024, np.uint8)
    assert f(5, buf.ctypes.data, buf.ctypes.data, 1, 32) == lean.LEAN_ERR_FORMAT
    assert f(0, None, buf.ctypes.data, 1, 32) == lean.LEAN_ERR_NULL
    assert f(0, buf.ctypes.data, buf.ctypes.data, 1, 33) == lean.LEAN_ERR_SHAPE
    for s in range(6):
        assert lean.status_str(s)


def test_device_status_codes_and_build_kind(lean):
    """LEAN_ERR_KERNEL_BOUNDS and LEAN_ERR_DEVICE are declared, described,
    and the product library is the release build (no index checks)."""
    import re
    hdr = open(os.path.join(ROOT, "include", "lean_qmatmul.h")).read()
    assert re.search(r"LEAN_ERR_KERNEL_BOUNDS\s*=\s*6", hdr)
    assert re.search(r"LEAN_ERR_DEVICE\s*=\s*7", hdr)
    assert lean.LEAN_ERR_KERNEL_BOUNDS == 6 and lean.LEAN_ERR_DEVICE == 7
    assert "LEAN_DEBUG" in lean.status_str(lean.LEAN_ERR_KERNEL_BOUNDS)
    assert "error word" in lean.status_str(lean.LEAN_ERR_DEVICE)
    assert lean.lean_debug_build() == 0


def test_library_keeps_its_own_statics(lean):
    """The library binds its own symbols and has no GNU-unique ones, so two
    builds loaded into one process (the release and the LEAN_DEBUG library)
    keep separate per-device caches."""
    import shutil
    import subprocess
    if not shutil.which("readelf"):
        pytest.skip("readelf not installed")
    lib = lib_build.LIB
    syms = subprocess.run(["readelf", "--dyn-syms", "-W", lib], capture_output=True, text=True).stdout
    assert "UNIQUE" not in syms
    dyn = subprocess.run(["readelf", "-d", lib], capture_output=True, text=True).stdout
    assert "SYMBOLIC" in dyn
