"""Plain fp64 CPU oracle for the block-quantized weight x activation product.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never calls it and shares no code with it.

The arithmetic lives in ``lean_oracle.c`` (scalar C, fp64): every weight is
decoded from its canonical block bytes and the dot product is summed in fp64.
This module only compiles that file with gcc and marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lean_oracle.c")
_LIB = os.path.join(_HERE, "liblean_oracle.so")
_lock = threading.Lock()
_lib = None

Q4_0, Q8_0, I8_B64, Q6_K = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile lean_oracle.c into liblean_oracle.so next to it (gcc, -O2)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    _gcc(_SRC, tmp)
    os.replace(tmp, _LIB)
    return _LIB


def _gcc(src: str, out: str) -> None:
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-Wall", "-Wextra", "-o", out, src, "-lm"], check=True)


def source() -> str:
    """Text of lean_oracle.c (the tests plant mistakes in copies of it)."""
    with open(_SRC) as f:
        return f.read()


def build_variant(src_text: str, out_path: str) -> str:
    """Compile C source text (a modified copy of lean_oracle.c, for the tests
    that check the pins catch planted mistakes) into the library out_path."""
    c_path = str(out_path) + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    _gcc(c_path, str(out_path))
    return str(out_path)


def _configure(lib):
    c_i64, c_int = ctypes.c_int64, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = ctypes.c_double
    lib.oracle_block_elems.argtypes = [c_int]
    lib.oracle_block_elems.restype = c_int
    lib.oracle_block_bytes.argtypes = [c_int]
    lib.oracle_block_bytes.restype = c_int
    lib.oracle_dequant.argtypes = [c_int, vp, c_i64, c_i64, vp]
    lib.oracle_dequant.restype = c_int
    lib.oracle_qmatmul.argtypes = [c_int, vp, vp, vp, vp, c_i64, c_i64, c_i64, c_int]
    lib.oracle_qmatmul.restype = c_int
    lib.oracle_qmatmul_pairs.argtypes = [c_int, vp, vp, c_i64, c_i64, c_i64, c_i64,
                                         vp, vp, vp, vp]
    lib.oracle_qmatmul_pairs.restype = c_int
    lib.oracle_quantize.argtypes = [c_int, vp, vp, c_i64, c_i64]
    lib.oracle_quantize.restype = c_int
    lib.oracle_double_to_fp16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_fp16.restype = c_int
    lib.oracle_quantize_x_int8.argtypes = [vp, vp, vp, c_i64, c_i64]
    lib.oracle_quantize_x_int8.restype = c_int
    lib.oracle_qmatmul_x_int8.argtypes = [c_int, vp, vp, vp, vp, c_i64, c_i64, c_i64]
    lib.oracle_qmatmul_x_int8.restype = c_int
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_swiglu.argtypes = [c_int, vp, vp, vp, vp, vp, vp, vp, vp, c_i64, c_i64]
    lib.oracle_swiglu.restype = c_int
    return lib


def load_library(path: str):
    """A ctypes handle on an oracle library built from (a copy of) lean_oracle.c."""
    return _configure(ctypes.CDLL(str(path)))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


class using:
    """Context manager: route this module's functions to another oracle
    library (load_library) for the duration of the block."""

    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def fp16_to_double(bits: int) -> float:
    return _load().oracle_fp16_to_double(bits)


def block_elems(fmt: int) -> int:
    return _load().oracle_block_elems(fmt)


def block_bytes(fmt: int) -> int:
    return _load().oracle_block_bytes(fmt)


def _check_w(fmt, W, N, K):
    be, bb = block_elems(fmt), block_bytes(fmt)
    if be == 0 or K % be:
        raise ValueError("bad format or K")
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if W.size != N * (K // be) * bb:
        raise ValueError("W has %d bytes, expected %d" % (W.size, N * (K // be) * bb))
    return W


def dequant(fmt: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Exact fp64 weights w[N][K] decoded from canonical blocks."""
    W = _check_w(fmt, W, N, K)
    w = np.empty((N, K), dtype=np.float64)
    if _load().oracle_dequant(fmt, _ptr(W), N, K, _ptr(w)):
        raise ValueError("oracle_dequant failed")
    return w


def qmatmul(fmt: int, W: np.ndarray, x: np.ndarray, N: int, K: int,
            threads: int = 1):
    """Return (y[M][N], bound[M][N]) in fp64 for canonical W and fp32 x[M][K]."""
    W = _check_w(fmt, W, N, K)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_qmatmul(fmt, _ptr(W), _ptr(x), _ptr(y), _ptr(b), N, K, M, threads)
    if rc:
        raise ValueError("oracle_qmatmul failed (%d)" % rc)
    return y, b


def qmatmul_pairs(fmt: int, W: np.ndarray, x: np.ndarray, N: int, K: int,
                  m_idx, n_idx):
    """(y, bound) for the selected output pairs (m_idx[i], n_idx[i]) only."""
    W = _check_w(fmt, W, N, K)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    P = m_idx.size
    y = np.empty(P, dtype=np.float64)
    b = np.empty(P, dtype=np.float64)
    rc = _load().oracle_qmatmul_pairs(fmt, _ptr(W), _ptr(x), N, K, x.shape[0], P,
                                      _ptr(m_idx), _ptr(n_idx), _ptr(y), _ptr(b))
    if rc:
        raise ValueError("oracle_qmatmul_pairs failed (%d)" % rc)
    return y, b


def double_to_fp16(v: float) -> int:
    """binary16 bits of the value nearest to v (ties to even), or -1."""
    return _load().oracle_double_to_fp16(float(v))


def quantize(fmt: int, w: np.ndarray, N: int, K: int) -> np.ndarray:
    """Canonical blocks of fp32 w[N][K] by the quantizer reading in
    lean_oracle.c (Q4_0, Q8_0, I8_B64); ValueError if it rejects the input."""
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(N, K)
    be, bb = block_elems(fmt), block_bytes(fmt)
    if be == 0 or K % be:
        raise ValueError("bad format or K")
    out = np.zeros(N * (K // be) * bb, dtype=np.uint8)
    if _load().oracle_quantize(fmt, _ptr(w), _ptr(out), N, K):
        raise ValueError("oracle_quantize rejected the input")
    return out


def quantize_x_int8(x: np.ndarray):
    """x[M][K] fp32 -> (codes int8[M][K], scales fp32[M][K/32]) by the
    activation-quantization reading in lean_oracle.c."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    M, K = x2.shape
    xq = np.empty((M, K), np.int8)
    sc = np.empty((M, K // 32), np.float32)
    if _load().oracle_quantize_x_int8(_ptr(x2), _ptr(xq), _ptr(sc), M, K):
        raise ValueError("K must be a positive multiple of 32")
    return xq, sc


def qmatmul_x_int8(fmt: int, W: np.ndarray, x: np.ndarray, N: int, K: int):
    """(y[M][N], bound[M][N]) in fp64 of the product with x quantized to int8
    per 32 elements (the reading in lean_oracle.c)."""
    W = _check_w(fmt, W, N, K)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_qmatmul_x_int8(fmt, _ptr(W), _ptr(x), _ptr(y), _ptr(b), N, K, M)
    if rc:
        raise ValueError("oracle_qmatmul_x_int8 failed (%d)" % rc)
    return y, b


def silu(t: float) -> float:
    """t / (1 + e^-t) in fp64."""
    return _load().oracle_silu(float(t))


def swiglu(fmt: int, Wg: np.ndarray, Wu: np.ndarray, x: np.ndarray, N: int, K: int):
    """h = silu(W_gate x) * (W_up x) for one x[K]; returns (h, g, u, bound_g,
    bound_u), each fp64 [N]."""
    Wg = _check_w(fmt, Wg, N, K)
    Wu = _check_w(fmt, Wu, N, K)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size != K:
        raise ValueError("x must have K elements")
    out = [np.empty(N, dtype=np.float64) for _ in range(5)]
    rc = _load().oracle_swiglu(fmt, _ptr(Wg), _ptr(Wu), _ptr(x), *[_ptr(a) for a in out], N, K)
    if rc:
        raise ValueError("oracle_swiglu failed (%d)" % rc)
    return tuple(out)
