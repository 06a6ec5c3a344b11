"""CPU oracle for paged decode attention over a tree-shaped, refcounted KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or runs
anything in this package.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.

The oracle is deliberately plain and slow:

* :mod:`oracle.attention` -- fp64 ``softmax(q K^T * scale) V`` for one decode
  query per branch, after gathering each branch's tokens through its block
  table into contiguous fp64 arrays ("The Reasoning Engine Meltdown", §2.1
  attention equation; "Dismantling the Memory Wall", PagedAttention section,
  ``BlockTable.get_block_for_token``).
* :mod:`oracle.allocator` -- a pure-Python model of the block pool: refcounted
  physical blocks, per-branch block tables, fork with copy-on-write of the last
  partial block, free, and eviction ordered by the importance score
  omega = branch_score / (depth + 1) ("The Reasoning Engine Meltdown", §5 and
  §6; RKSC summary, §2.C RSBCM).
* :mod:`oracle.fp8` -- FP8 (E4M3) KV storage: the element format from its
  definition, one power-of-two scale per (block, kv-head) and tensor, block
  writes with re-encoding when the scale grows, and decode over the
  dequantised values (a reading: the pages only name FP8 KV quantisation,
  "The Reasoning Engine Meltdown", §9).
* :mod:`oracle.radix` -- the token-keyed radix prefix index ("Dismantling the
  Memory Wall", RadixAttention section).
* :mod:`oracle.brute` -- a scalar pure-Python restatement used only on tiny
  inputs as an extra cross-check of the vectorised code.

It shares no code, header, table or helper with the CUDA library; the only
thing both sides consume is the seeded synthetic input produced by
``paged_kv_cache_attn_gb300.workloads`` (which holds none of the method's
arithmetic).

Parity pins (tests/test_oracle_*.py): closed forms (L = 1, identical keys,
a dominant key, two-token sigmoid), invariants (physical-block permutation,
shared vs private prefix layout, key-order permutation, score shift, linearity
in V), the pages' KV-size worked example, the pages' page-table diagram and
the allocator rules; for FP8, PyTorch's independent float8_e4m3fn type, hand-worked
codes, the scale's defining inequalities, the 3-bit-mantissa error bound and a
derived bound on the attention output.  No oracle function is "parity unpinned".
"""
