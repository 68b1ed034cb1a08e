"""Build ``liblean_qmatmul.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  No cmake, no torch extension machinery: the
library is a plain C ABI (``include/lean_qmatmul.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "liblean_qmatmul.so")
BUILD = os.path.join(ROOT, "_build")
# the LEAN_DEBUG build: every kernel checks its global-memory indices
# (csrc/debug.cuh); same ABI, its own objects and library
DEBUG_LIB = os.path.join(HERE, "liblean_qmatmul_debug.so")
DEBUG_BUILD = os.path.join(ROOT, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fno-gnu-unique and -Bsymbolic (at link time): the library keeps its own
# copy of every function-local static (per-device caches such as "shared-memory
# limit raised for this kernel") even when another build of it (the LEAN_DEBUG
# one) is loaded into the same process; GNU-unique symbols would otherwise be
# shared process-wide and one build would skip the other's setup
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-Xcompiler", "-fno-gnu-unique", "--expt-relaxed-constexpr"] + ARCH
SOURCES = ["lean_qmatmul.cu", "pack.cpp", "qmm_q4_0.cu", "qmm_q8_0.cu", "qmm_i8_b64.cu", "qmm_q6_k.cu",
           "qmm_fixed_ws.cu"]
# host-only helpers (no CUDA), compiled by the host C++ compiler
HOST = os.path.join(HERE, "host")
HOST_SOURCES = ["quant.cpp"]
HOST_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-ffp-contract=off", "-pthread", "-fno-gnu-unique"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(HOST, f) for f in os.listdir(HOST)]
    inc = os.path.join(ROOT, "include")
    files += [os.path.join(inc, f) for f in os.listdir(inc)]
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def _compile_host(src: str, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, "host_" + os.path.basename(src) + ".o")
    cxx = os.environ.get("CXX") or shutil.which("g++") or "c++"
    cmd = [cxx] + HOST_FLAGS + ["-c", os.path.join(HOST, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("host compile failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build(force: bool = False, verbose: bool = False, extra=(), debug: bool = False) -> str:
    """Compile every source for sm_103a and link liblean_qmatmul.so (debug:
    with -DLEAN_DEBUG into liblean_qmatmul_debug.so)."""
    lib, build_dir = (DEBUG_LIB, DEBUG_BUILD) if debug else (LIB, BUILD)
    if debug:
        extra = tuple(extra) + ("-DLEAN_DEBUG",)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES) + len(HOST_SOURCES)) as ex:
        dev = [ex.submit(_compile, s, extra, build_dir) for s in SOURCES]
        host = [ex.submit(_compile_host, s, build_dir) for s in HOST_SOURCES]
        objs = [f.result() for f in dev + host]
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-Xlinker", "-Bsymbolic", "-o", tmp] + objs + ["-lcudart", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else (), debug="--debug" in sys.argv)
