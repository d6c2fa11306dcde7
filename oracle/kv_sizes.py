"""Closed forms for KV-cache sizes and paged-allocation waste.

* Per-token KV bytes = 2 (K and V) x n_layers x n_kv_heads x head_dim x
  dtype_bytes ("Modern AI Infrastructure and Agentic System Design", 9.1
  "The key and value cache"; "Inference serving: the KV-cache machine",
  section "The KV cache: attention's memory bill, derived").
* A paged sequence of n tokens holds ceil(n / block_size) blocks, so at most
  block_size - 1 slots of its last block are empty ("PagedAttention vs
  Traditional KV Cache", Section 5 "Memory Fragmentation: Before vs After";
  Section 7 "Trade-offs and Limitations", block-size sensitivity).
"""
from __future__ import annotations

import math


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def kv_cache_bytes(n_layers, n_kv_heads, head_dim, dtype_bytes, seq_len, batch) -> int:
    return kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype_bytes) * seq_len * batch


def blocks_for(n_tokens: int, block_size: int) -> int:
    return int(math.ceil(n_tokens / block_size)) if n_tokens > 0 else 0


def tail_waste_slots(n_tokens: int, block_size: int) -> int:
    return blocks_for(n_tokens, block_size) * block_size - n_tokens


def max_waste_fraction(block_size: int, avg_seq_len: float) -> float:
    """Worst case: the last block holds one token, block_size - 1 slots empty."""
    return (block_size - 1) / avg_seq_len


def decode_kv_read_bytes(context_lens, n_kv_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Unique K+V bytes one decode step of one layer reads: every valid token's
    K and V rows for every KV head."""
    return 2 * n_kv_heads * head_dim * dtype_bytes * int(sum(max(int(c), 0) for c in context_lens))
