"""Attention over a paged KV cache, hand-written CUDA for GB300 (sm_103a).

The compute lives in ``libpagedkv.so`` (C ABI declared in ``include/pagedkv.h``);
``paged_kv_flash_gb300.pagedkv`` is the thin ctypes binding over it.  The
binding is imported lazily so that the seeded input generators in
``paged_kv_flash_gb300.workloads`` stay usable without a built library.
"""

__all__ = ["pagedkv", "workloads"]


def __getattr__(name):
    if name == "pagedkv":
        from . import pagedkv
        return pagedkv
    raise AttributeError(name)
