"""GB300 paged-KV decode attention over a tree-shaped, refcounted KV cache.

* ``include/pagedkv.h`` -- the C ABI (pool, branches, fork with copy-on-write,
  free, eviction by omega = score / (depth + 1), batch builder, decode plan,
  ``paged_decode_attn``).
* ``paged_kv_cache_attn_gb300.binding`` -- the ctypes binding (same names).
* ``paged_kv_cache_attn_gb300.harness`` -- replays a synthetic workload
  through the binding.
* ``paged_kv_cache_attn_gb300.workloads`` -- seeded synthetic workloads.
* ``paged_kv_cache_attn_gb300.build`` -- builds ``_build/libpagedkv.so``.

Submodules are imported on demand so that ``workloads`` can be used without
the compiled library.
"""
