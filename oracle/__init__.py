"""fp64 CPU oracle for paged decode attention and its cache-maintenance steps.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) imports, calls or links anything here. The only users are the
tests under ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``. The oracle shares no code with the CUDA path; both sides take
their inputs from the seeded generator in ``workloads/``.

What each function computes is the plain definition the pages give:

* ``attention.paged_decode`` / ``attention.paged_prefill`` - gather each
  sequence's K/V through its block table into a contiguous array, then
  softmax(q K^T * scale) V in fp64 ("KV Cache Explained Like You're an LLM
  Engineer", section "Transformer Attention: A Quick Refresher";
  "LLM Inference Optimization: KV-Cache, PagedAttention, and GPU Memory
  Efficiency", section "PagedAttention: OS Concepts Meet GPU Memory").
* ``cache_ops.reshape_and_cache`` / ``cache_ops.copy_blocks`` - scatter of new
  tokens to their slots, and the copy-on-write block copy.
* ``block_manager.BlockManagerModel`` - free list, refcounts, fork and
  copy-on-write ("Inference serving: the KV-cache machine", section "Paged KV:
  virtual memory for tokens"; "Modern AI Infrastructure and Agentic System
  Design", 9.1 "The key and value cache").
* ``kv_sizes`` - the per-token KV-bytes closed form.

Every function is pinned by tests in ``tests/test_oracle_*.py`` to something
other than itself (a library routine on a special case, closed forms, values
the pages print, invariants). No function here is "parity unpinned".
"""
from . import attention, block_manager, cache_ops, kv_sizes  # noqa: F401
from .bf16 import bf16_bits_to_f64  # noqa: F401
