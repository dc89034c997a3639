"""CacheGen KV-cache codec for GB300 (sm_103a).

The codec itself is the C ABI in include/cachegen.h, implemented by the CUDA
library libcachegen_gb300.so built from csrc/ (``python -m
kv_cache_compression_cg_gb300.build``). ``capi`` is the ctypes binding with the
same function names; ``codec`` wraps it for PyTorch tensors (PyTorch supplies
device memory and streams only). ``synth`` is the seeded input generator;
``shard`` splits a tensor over ranks by chunk ranges and joins the outputs;
``stream`` pipelines host-to-device copies, coding and copies back by chunk runs.
"""
from __future__ import annotations

__all__ = ["capi", "codec", "synth", "build", "shard", "stream"]


def __getattr__(name):
    import importlib
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
