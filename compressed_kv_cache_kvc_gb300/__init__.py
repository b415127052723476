"""Compressed-KV decode step for GB300 (sm_103a).

The compute lives in the CUDA library ``libkvc.so`` (C ABI: ``include/kvc.h``);
``KVCache`` is a thin binding that passes device pointers and the torch CUDA
stream to it.
"""
from . import workloads  # noqa: F401

__all__ = ["KVCache", "workloads"]


def __getattr__(name):
    if name == "KVCache":
        from .cache import KVCache
        return KVCache
    raise AttributeError(name)
