"""Cache-maintenance oracle: new-token scatter and copy-on-write block copy.

* reshape_and_cache: every decode step appends the new token's K and V to the
  cache ("KV Cache Explained Like You're an LLM Engineer", section "What KV
  Cache Stores"). In a paged cache the token's place is a slot, i.e. physical
  block table[pos // block_size] at offset pos % block_size ("Inference
  serving: the KV-cache machine", section "Paged KV: virtual memory for
  tokens": token 41 goes to table[2]). Slot encoding used by the library:
  slot = block * block_size + offset; a negative slot means "skip this row".
* copy_blocks: a write to a block shared by several sequences first copies the
  block into a fresh one ("Modern AI Infrastructure and Agentic System
  Design", 9.1 "The key and value cache", the copy-on-write figure; "LLM
  Inference Optimization: KV-Cache, PagedAttention, and GPU Memory
  Efficiency", section "PagedAttention: OS Concepts Meet GPU Memory": only the
  diverging block gets copied). The copy moves every KV head and every slot
  of the block, for K and for V.

* swap_out / swap_in: preemption by swapping moves a sequence's private
  blocks to host memory and later back into any free blocks ("Modern AI
  Infrastructure and Agentic System Design", 9.1, part "Batching and the
  scheduler"; "Inference serving: the KV-cache machine", section "Paged KV:
  virtual memory for tokens"). The host copy holds the blocks in the order
  given, each with the pool's block layout.

All are bit copies; the oracle works on the raw bit patterns and returns new
arrays (the inputs are not modified).
"""
from __future__ import annotations

import numpy as np


def slot_to_block_offset(slot: int, block_size: int):
    return int(slot) // block_size, int(slot) % block_size


def reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping):
    """k_new, v_new [T][n_kv_heads][head_dim]; pools [blocks][n_kv_heads][bs][D].

    Row t goes to (block, offset) = divmod(slot_mapping[t], bs) for every KV
    head; rows with a negative slot are skipped.
    """
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    bs = kp.shape[2]
    for t, s in enumerate(np.asarray(slot_mapping)):
        if int(s) < 0:
            continue
        blk, off = slot_to_block_offset(int(s), bs)
        kp[blk, :, off, :] = k_new[t]
        vp[blk, :, off, :] = v_new[t]
    return kp, vp


def copy_blocks(k_pool, v_pool, block_mapping):
    """block_mapping [n][2] of (src, dst): dst's whole block := src's block.

    Pairs are applied in order; a destination is expected to be a fresh block
    (not a source of another pair).
    """
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for src, dst in np.asarray(block_mapping).reshape(-1, 2):
        kp[int(dst)] = kp[int(src)]
        vp[int(dst)] = vp[int(src)]
    return kp, vp


def swap_out(k_pool, v_pool, block_ids):
    """Host copies [n][n_kv_heads][bs][D] of pool blocks block_ids, in order."""
    ids = [int(b) for b in np.asarray(block_ids)]
    return (np.array([np.asarray(k_pool)[b] for b in ids]).reshape((len(ids),) + np.asarray(k_pool).shape[1:]),
            np.array([np.asarray(v_pool)[b] for b in ids]).reshape((len(ids),) + np.asarray(v_pool).shape[1:]))


def swap_in(host_k, host_v, k_pool, v_pool, block_ids):
    """Pool block block_ids[i] := host block i (new arrays returned)."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for i, b in enumerate(np.asarray(block_ids)):
        kp[int(b)] = host_k[i]
        vp[int(b)] = host_v[i]
    return kp, vp
