"""Paged-KV decode attention for GB300 (sm_103a).

The library is a C ABI (``include/pa.h``, ``libpa.so`` built from ``csrc/``)
with hand-written CUDA kernels.  ``paged_kv_decode_07_gb300.pa`` is the thin
ctypes binding with the same entry-point names; it is loaded lazily, so
importing the synthetic-workload generators (``.workloads``) never touches
the CUDA library.  Calling any entry point without the built library raises.
"""
from __future__ import annotations

import importlib

_SUBMODULES = ("pa", "workloads", "build")
_API = ("decode", "verify", "merge", "dequant_gather", "workspace_bytes", "read_error",
        "status_string", "KvCache", "PaError", "library_path")


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    if name in _API:
        return getattr(importlib.import_module(f"{__name__}.pa"), name)
    raise AttributeError(name)
