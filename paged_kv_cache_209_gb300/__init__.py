"""pkv: paged KV-cache decode attention for GB300 (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA behind a C ABI declared
in ``include/pkv.h``). ``paged_kv_cache_209_gb300.pkv`` is the thin ctypes
binding with the same function names; importing this package does not load
the library, so ``workloads`` can be used without a GPU.
"""

__all__ = ["pkv", "workloads"]
