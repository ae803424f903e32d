"""GB300-native DKV decode attention over an anchor + low-rank differential KV cache.

The compute path lives in the CUDA library ``libdkv.so`` (built from ``csrc/``)
and is reached through :mod:`compressed_kv_cache_dkv_gb300.dkv`, a thin ctypes
binding.  Importing this package does not load the library; the binding
raises when it is used without the library.
"""
__all__ = ["synth"]
