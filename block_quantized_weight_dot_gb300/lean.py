"""ctypes binding of ``liblean_qmatmul.so`` (C ABI in ``include/lean_qmatmul.h`` and
``include/lean_quant.h``).

Argument marshalling only: every computation of the product runs in the CUDA
library.  Functions keep the C names.  Buffers may be given as torch tensors
(their ``data_ptr()`` is passed), numpy arrays (host calls only) or raw integer
addresses.  A non-OK status raises :class:`LeanError`.  If the library has not
been built the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblean_qmatmul.so")
# the LEAN_DEBUG build of the same ABI (build.build(debug=True)): every kernel
# checks its global-memory indices; for test runs (open_library / use_library)
DEBUG_LIB_PATH = os.path.join(_HERE, "liblean_qmatmul_debug.so")

LEAN_Q4_0, LEAN_Q8_0, LEAN_I8_B64, LEAN_Q6_K = 0, 1, 2, 3
(LEAN_OK, LEAN_ERR_FORMAT, LEAN_ERR_SHAPE, LEAN_ERR_NULL, LEAN_ERR_ALIGN, LEAN_ERR_CUDA,
 LEAN_ERR_KERNEL_BOUNDS, LEAN_ERR_DEVICE) = range(8)
LEAN_FLAG_EARLY_WEIGHTS = 1
LEAN_FLAG_X_PLANES = 2
LEAN_FLAG_STREAM = 4
LEAN_FLAG_X_INT8 = 8

# every symbol the header declares, with (restype, argtypes)
_i64, _int, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "lean_block_elems": (_int, [_int]),
    "lean_block_bytes": (_i64, [_int]),
    "lean_canonical_bytes": (_i64, [_int, _i64, _i64]),
    "lean_packed_bytes": (_i64, [_int, _i64, _i64]),
    "lean_pack": (_int, [_int, _vp, _vp, _i64, _i64]),
    "lean_unpack_canonical": (_int, [_int, _vp, _vp, _i64, _i64]),
    "lean_dequant": (_int, [_int, _vp, _vp, _i64, _i64, _vp]),
    "lean_embed_rows": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "lean_qmatmul_swiglu": (_int, [_int, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_uint, _vp]),
    "lean_qmatmul": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "lean_qmatmul_ex": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_uint, _vp]),
    "lean_qmatmul_workspace_bytes": (_i64, [_int, _i64, _i64, _i64]),
    "lean_tensor_core_min_m": (_int, [_int]),
    "lean_qmatmul_ws": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_uint, _vp, _i64,
                               _vp]),
    "lean_batch_workspace_bytes": (_i64, [_int, _int, _vp]),
    "lean_qmatmul_batch": (_int, [_int, _int, _vp, ctypes.c_uint, _vp, _i64, _vp]),
    "lean_device_error": (ctypes.c_uint, [_int]),
    "lean_device_status": (_int, [_int]),
    "lean_debug_build": (_int, []),
    "lean_wait_selftest": (_int, [ctypes.c_uint, _vp]),
    "lean_quantize": (_int, [_int, _vp, _vp, _i64, _i64, _int]),
    "lean_qmatmul_fixed_ws": (_int, [_int, _vp, _vp, _vp, _i64, _i64, ctypes.c_uint, _vp]),
    "lean_fixed_workspace_bytes": (_i64, []),
    "lean_status_str": (ctypes.c_char_p, [_int]),
}
LEAN_MAX_BATCH = 256


class lean_problem(ctypes.Structure):
    """One product of a batch: device pointers and its shape (C struct lean_problem)."""
    _fields_ = [("W", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class LeanError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, status_str(status), status))


def open_library(path: str):
    """A ctypes handle on a build of this ABI (the product library or its
    LEAN_DEBUG build), with every declared signature set."""
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("liblean_qmatmul.so is not built: run "
                          "`python -c \"import __graft_entry__ as g; g.build()\"`")
    return open_library(LIB_PATH)


_lib = _load()


def use_library(lib):
    """Route every call of this module through `lib` (a handle from
    open_library); returns the handle used until now."""
    global _lib
    prev, _lib = _lib, lib
    return prev


def _addr(buf):
    """Address of a buffer: torch tensor, numpy array, int or None."""
    if buf is None:
        return None
    if isinstance(buf, int):
        return buf
    if isinstance(buf, np.ndarray):
        return buf.ctypes.data
    if hasattr(buf, "data_ptr"):
        return buf.data_ptr()
    raise TypeError("unsupported buffer type %r" % type(buf))


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def _check(fn, status):
    if status != LEAN_OK:
        raise LeanError(fn, status)


def status_str(status: int) -> str:
    return _lib.lean_status_str(status).decode()


lean_status_str = status_str


def lean_block_elems(fmt: int) -> int:
    return _lib.lean_block_elems(fmt)


def lean_block_bytes(fmt: int) -> int:
    return _lib.lean_block_bytes(fmt)


def lean_canonical_bytes(fmt: int, N: int, K: int) -> int:
    return _lib.lean_canonical_bytes(fmt, N, K)


def lean_packed_bytes(fmt: int, N: int, K: int) -> int:
    return _lib.lean_packed_bytes(fmt, N, K)


def lean_pack(fmt: int, canon, N: int, K: int, packed=None) -> np.ndarray:
    """Canonical host bytes -> packed host bytes (a new uint8 array unless given)."""
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    nb = lean_packed_bytes(fmt, N, K)
    if nb < 0:
        raise LeanError("lean_pack", LEAN_ERR_SHAPE)
    if canon.size != lean_canonical_bytes(fmt, N, K):
        raise ValueError("canonical buffer has %d bytes, expected %d"
                         % (canon.size, lean_canonical_bytes(fmt, N, K)))
    if packed is None:
        packed = np.empty(nb, dtype=np.uint8)
    _check("lean_pack", _lib.lean_pack(fmt, _addr(canon), _addr(packed), N, K))
    return packed


def lean_unpack_canonical(fmt: int, packed, N: int, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size != lean_packed_bytes(fmt, N, K):
        raise ValueError("packed buffer has the wrong size")
    canon = np.empty(lean_canonical_bytes(fmt, N, K), dtype=np.uint8)
    _check("lean_unpack_canonical", _lib.lean_unpack_canonical(fmt, _addr(packed), _addr(canon), N, K))
    return canon


def lean_dequant(fmt: int, W_packed_dev, w_dev, N: int, K: int, stream=None) -> None:
    _check("lean_dequant", _lib.lean_dequant(fmt, _addr(W_packed_dev), _addr(w_dev), N, K,
                                             _stream(stream)))


def lean_embed_rows(fmt: int, W_packed_dev, ids_dev, out_dev, n_ids: int, N: int, K: int,
                    stream=None) -> None:
    """out[i][k] = w[ids[i]][k] (an embedding lookup); ids: int32 device tensor."""
    _check("lean_embed_rows", _lib.lean_embed_rows(fmt, _addr(W_packed_dev), _addr(ids_dev),
                                                   _addr(out_dev), n_ids, N, K, _stream(stream)))


def lean_qmatmul_swiglu(fmt: int, W_gate_dev, W_up_dev, x_dev, h_dev, N: int, K: int,
                        flags: int = 0, stream=None) -> None:
    """h = silu(W_gate x) * (W_up x) in one launch (M = 1)."""
    _check("lean_qmatmul_swiglu", _lib.lean_qmatmul_swiglu(
        fmt, _addr(W_gate_dev), _addr(W_up_dev), _addr(x_dev), _addr(h_dev), N, K, flags,
        _stream(stream)))


def lean_qmatmul(fmt: int, W_packed_dev, x_dev, y_dev, N: int, K: int, M: int,
                 stream=None) -> None:
    """y[M][N] = x[M][K] . W[N][K]^T on the device, asynchronously on `stream`."""
    _check("lean_qmatmul", _lib.lean_qmatmul(fmt, _addr(W_packed_dev), _addr(x_dev),
                                             _addr(y_dev), N, K, M, _stream(stream)))


def lean_qmatmul_ex(fmt: int, W_packed_dev, x_dev, y_dev, N: int, K: int, M: int,
                    flags: int = 0, stream=None) -> None:
    """lean_qmatmul with launch flags (LEAN_FLAG_EARLY_WEIGHTS, LEAN_FLAG_X_PLANES)."""
    _check("lean_qmatmul_ex", _lib.lean_qmatmul_ex(fmt, _addr(W_packed_dev), _addr(x_dev),
                                                   _addr(y_dev), N, K, M, flags, _stream(stream)))


def lean_qmatmul_workspace_bytes(fmt: int, N: int, K: int, M: int) -> int:
    return _lib.lean_qmatmul_workspace_bytes(fmt, N, K, M)


def lean_tensor_core_min_m(fmt: int) -> int:
    """Rows of x from which the product of format fmt runs on the tensor cores."""
    return _lib.lean_tensor_core_min_m(fmt)


def lean_qmatmul_ws(fmt: int, W_packed_dev, x_dev, y_dev, N: int, K: int, M: int,
                    flags: int = 0, workspace=None, workspace_bytes: int = 0,
                    stream=None) -> None:
    """lean_qmatmul with flags and a caller-owned, once-zeroed device workspace."""
    _check("lean_qmatmul_ws", _lib.lean_qmatmul_ws(fmt, _addr(W_packed_dev), _addr(x_dev),
                                                   _addr(y_dev), N, K, M, flags,
                                                   _addr(workspace), workspace_bytes,
                                                   _stream(stream)))


def make_problems(items):
    """ctypes array of lean_problem from (W, x, y, N, K) tuples."""
    arr = (lean_problem * len(items))()
    for i, (W, x, y, N, K) in enumerate(items):
        arr[i] = lean_problem(_addr(W), _addr(x), _addr(y), N, K)
    return arr


def lean_batch_workspace_bytes(fmt: int, problems) -> int:
    return _lib.lean_batch_workspace_bytes(fmt, len(problems), ctypes.cast(problems, _vp))


def lean_qmatmul_batch(fmt: int, problems, flags: int = 0, workspace=None,
                       workspace_bytes: int = 0, stream=None) -> None:
    """Independent M = 1 products in one launch; `problems` from make_problems()."""
    _check("lean_qmatmul_batch", _lib.lean_qmatmul_batch(fmt, len(problems),
                                                         ctypes.cast(problems, _vp), flags,
                                                         _addr(workspace), workspace_bytes,
                                                         _stream(stream)))


def lean_qmatmul_fixed_ws(fmt: int, W_packed_dev, x_dev, y_dev, N: int, K: int, flags: int = 0,
                          stream=None) -> None:
    """M = 1 product whose scratch is the library's own fixed device array (no
    allocation by the caller; calls overlapping on the GPU must be serialised)."""
    _check("lean_qmatmul_fixed_ws", _lib.lean_qmatmul_fixed_ws(fmt, _addr(W_packed_dev),
                                                               _addr(x_dev), _addr(y_dev), N, K,
                                                               flags, _stream(stream)))


def lean_fixed_workspace_bytes() -> int:
    return _lib.lean_fixed_workspace_bytes()


def lean_device_error(clear: bool = True) -> int:
    """Device error word (non-zero: a kernel's bounded wait timed out)."""
    return _lib.lean_device_error(1 if clear else 0)


def lean_quantize(fmt: int, w, N: int, K: int, threads: int = 0):
    """Canonical blocks (uint8 array, ready for lean_pack) of fp32 w[N][K]
    quantized on the host to Q4_0, Q8_0 or I8_B64 (rule in lean_quant.h)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.size != N * K:
        raise ValueError("w has %d elements, expected %d" % (w.size, N * K))
    nbytes = lean_canonical_bytes(fmt, N, K)
    out = np.zeros(max(nbytes, 1), dtype=np.uint8)  # a bad shape is reported by the call
    _check("lean_quantize", _lib.lean_quantize(fmt, w.ctypes.data, out.ctypes.data, N, K,
                                                threads))
    return out[:nbytes]


def lean_device_status(clear: bool = True) -> int:
    """The device error word as a status (LEAN_OK, LEAN_ERR_KERNEL_BOUNDS,
    LEAN_ERR_DEVICE or LEAN_ERR_CUDA); returned, not raised."""
    return _lib.lean_device_status(1 if clear else 0)


def lean_debug_build() -> int:
    return _lib.lean_debug_build()


def lean_wait_selftest(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test: a block waits on a barrier nothing
    completes, gives up after limit_us and sets bit 8 of the error word."""
    _check("lean_wait_selftest", _lib.lean_wait_selftest(limit_us, _stream(stream)))


# ---- torch conveniences (device memory via PyTorch; compute via the library) ----

def upload_packed(fmt: int, canon, N: int, K: int, device="cuda"):
    """Pack canonical host bytes and copy them to a new uint8 device tensor."""
    import torch
    packed = lean_pack(fmt, canon, N, K)
    return torch.from_numpy(packed).to(device)


def qmatmul(fmt: int, W_packed_dev, x, N: int, K: int, out=None, stream=None):
    """Allocate y (or use `out`) and run lean_qmatmul; x is a [M, K] fp32 cuda tensor."""
    import torch
    x = x.contiguous()
    M = x.numel() // K
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    lean_qmatmul(fmt, W_packed_dev, x, y, N, K, M, stream)
    return y
