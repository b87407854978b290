"""Paged-KV decode attention for GB300 (sm_103a).

The library is a C ABI (``include/pa.h``, ``libpa.so`` built from ``csrc/``)
with hand-written CUDA kernels.  ``paged_kv_decode_07_gb300.pa`` is the thin
ctypes binding with the same entry-point names; it is loaded lazily, so
importing the synthetic-workload generators (``.workloads``) never touches
the CUDA library.  Calling any entry point without the built library raises.
"""
from __future__ import annotations

__all__ = ["pa", "workloads"]


def __getattr__(name):
    if name in ("pa", "workloads"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    # convenience: paged_kv_decode_07_gb300.decode(...) etc.
    from . import pa as _pa
    if hasattr(_pa, name):
        return getattr(_pa, name)
    raise AttributeError(name)
