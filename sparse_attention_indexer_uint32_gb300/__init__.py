"""GB300-native top-k + page-table transform for sparse-attention indexers.

The compute lives in ``libtopkidx.so`` (hand-written sm_103a CUDA, C ABI in
``include/topkidx.h``).  ``_lib`` is its ctypes binding with the C names;
``api`` adds tensor-allocating conveniences on top.  Importing the binding
raises if the library has not been built (there is no CPU fallback).
"""
from __future__ import annotations

__all__ = ["build", "workloads"]


def __getattr__(name):
    # The binding loads the CUDA library, so it is imported on first use only.
    if name in ("_lib", "api"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
