"""GB300-native paged KV cache hot path: kv_store, paged prefill, paged decode.

The compute lives in hand-written CUDA kernels for sm_103a behind a C ABI
(``include/pagedkv.h``, built into ``libpagedkv.so`` next to this file).
``paged_kv_cache_303_gb300.ops`` is a thin ctypes binding over that ABI that
takes torch CUDA tensors; it only marshals pointers, sizes and the stream.
There is no CPU fallback: every call fails loudly if the library is missing.
"""
import importlib

__all__ = ["ops", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
