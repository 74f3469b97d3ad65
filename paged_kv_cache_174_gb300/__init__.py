"""GB300-native attention over a paged KV cache.

The compute lives in ``libpagedattn.so`` (hand-written CUDA for sm_103a behind
a C ABI, declared in ``include/pagedattn.h``).  ``paged_kv_cache_174_gb300.ops``
is the thin Python binding over it; ``workloads`` draws seeded synthetic
inputs; ``host`` holds the block allocator and the continuous-batching step
driver that generate multi-step workloads.

Importing this package does not load the CUDA library; the first call into
``ops`` does, and raises if the library is missing.
"""

__all__ = ["ops", "workloads", "host"]
