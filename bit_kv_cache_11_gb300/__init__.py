"""GB300-native low-bit KV cache: per-channel key / per-token value
quantization with an fp16 tail, and split-K decode attention over the packed
cache.

The compute path is the CUDA library ``libkvq.so`` (C ABI in
``include/kvq.h``); ``bit_kv_cache_11_gb300.kvq`` is its thin ctypes binding
and raises at import time when the library is missing.  ``synth`` (seeded
inputs) imports without it.
"""
from __future__ import annotations

import importlib

__all__ = ["kvq", "synth", "build"]


def __getattr__(name):
    if name in ("kvq", "synth", "build"):
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
