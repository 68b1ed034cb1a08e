"""GB300 (sm_103a) block-quantized weight x activation product.

The compute path is the CUDA library ``liblean_qmatmul.so`` built from
``csrc/``; :mod:`.lean` is its thin ctypes binding (argument marshalling only).
The binding is loaded on first use and raises if the library is missing: there
is no CPU fallback.
"""
import importlib

from .synthetic import Q4_0, Q8_0, I8_B64, Q6_K  # noqa: F401


def __getattr__(name):
    # Load the CUDA binding lazily so that importing the synthetic-input module
    # does not require the compiled library.
    if name.startswith("__"):
        raise AttributeError(name)
    if name in ("lean", "build", "synthetic"):
        return importlib.import_module("." + name, __name__)
    return getattr(importlib.import_module(".lean", __name__), name)
