"""Attention over a paged KV cache, hand-written CUDA for GB300 (sm_103a).

The compute lives in ``libpagedkv.so`` (C ABI declared in ``include/pagedkv.h``);
``paged_kv_flash_gb300.pagedkv`` is the thin ctypes binding over it and loads
the library when imported.  ``paged_kv_flash_gb300.workloads`` holds the
seeded synthetic input generators and needs no built library.
"""
