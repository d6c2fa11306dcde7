"""fp64 paged attention oracle: gather through the block table, then attend.

Sources (cited by page title and section):
* "LLM Inference Optimization: KV-Cache, PagedAttention, and GPU Memory
  Efficiency", section "PagedAttention: OS Concepts Meet GPU Memory": a block
  table maps a logical position to (table[pos // block_size], pos % block_size),
  and the kernel loads K and V for the sequence's blocks and accumulates the
  attention. Paging changes only where a token's K/V is stored, so the result
  is the dense attention over the same tokens.
* "KV Cache Explained Like You're an LLM Engineer", section "Transformer
  Attention: A Quick Refresher": Attention(Q_i, K, V) = softmax(Q_i K^T / sqrt(d_k)) V;
  section "What KV Cache Stores": the new query attends to all cached keys
  including the one just appended.
* "What Happens Inside an LLM During Inference: Tokens, KV Cache, and GPU
  Execution Explained", section "Self-Attention Mechanism" (its
  scaled-dot-product attention listing): positions with mask 0
  are excluded from the softmax; a causal mask lets position i see j <= i.
* Grouped-query attention: a KV head serves a group of query heads
  ("Inference serving: the KV-cache machine", section "The KV cache:
  attention's memory bill, derived"). Reading taken: query head h uses KV head
  h // (n_heads // n_kv_heads), i.e. contiguous groups.

Steps follow the plain definition; there is no blocking, online rescaling or
reordering here. Each score is an fp64 dot product, the softmax subtracts the
row maximum before exp (a mathematical identity), and the output is the
p-weighted sum of V divided by the sum of p.

Layouts: pools [num_blocks][n_kv_heads][block_size][head_dim] (bf16 bits or
float), q [n][n_heads][head_dim], tables [n_seqs][max_blocks] int.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f64


def _as_f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def gather_kv(pool: np.ndarray, table_row: np.ndarray, n_tokens: int) -> np.ndarray:
    """Contiguous [n_tokens][n_kv_heads][head_dim] view of one sequence.

    Logical token t lives in physical block table_row[t // block_size] at
    offset t % block_size.
    """
    pool = np.asarray(pool)
    bs = pool.shape[2]
    out = np.empty((n_tokens, pool.shape[1], pool.shape[3]), dtype=pool.dtype)
    for t in range(n_tokens):
        out[t] = pool[int(table_row[t // bs]), :, t % bs, :]
    return out


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q . k^T * scale) . v for one query vector and one head, fp64.

    q [D], k [T][D], v [T][D] -> [D]. T == 0 gives a zero vector.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    if k.shape[0] == 0:
        return np.zeros(q.shape[-1], dtype=np.float64)
    s = (k @ q) * float(scale)
    p = np.exp(s - s.max())
    return (p @ v) / p.sum()


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale) -> np.ndarray:
    """Single-query attention for every sequence over its paged cache.

    q [B][H][D]; returns fp64 out [B][H][D]. context_lens[b] counts every
    valid token of sequence b (including the one written this step); a
    context length <= 0 gives a zero row.
    """
    q = np.asarray(q)
    B, H, D = q.shape
    Hk = np.asarray(k_pool).shape[1]
    g = H // Hk
    out = np.zeros((B, H, D), dtype=np.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n <= 0:
            continue
        kc = _as_f64(gather_kv(k_pool, block_tables[b], n))
        vc = _as_f64(gather_kv(v_pool, block_tables[b], n))
        for h in range(H):
            kh = h // g
            out[b, h] = attend(q[b, h], kc[:, kh, :], vc[:, kh, :], scale)
    return out


def paged_decode_rows(q, k_pool, v_pool, block_tables, context_lens, scale, rows):
    """paged_decode for a subset of (seq, head) pairs; returns {(b, h): out[D]}."""
    q = np.asarray(q)
    H = q.shape[1]
    Hk = np.asarray(k_pool).shape[1]
    g = H // Hk
    res = {}
    cache = {}
    for b, h in rows:
        b, h = int(b), int(h)
        n = int(context_lens[b])
        if n <= 0:
            res[(b, h)] = np.zeros(q.shape[2])
            continue
        key = (b, h // g)
        if key not in cache:
            kc = _as_f64(gather_kv(np.asarray(k_pool)[:, h // g:h // g + 1], block_tables[b], n))
            vc = _as_f64(gather_kv(np.asarray(v_pool)[:, h // g:h // g + 1], block_tables[b], n))
            cache[key] = (kc[:, 0, :], vc[:, 0, :])
        kc, vc = cache[key]
        res[(b, h)] = attend(q[b, h], kc, vc, scale)
    return res


def paged_decode_window(q, k_pool, v_pool, block_tables, context_lens, scale, window) -> np.ndarray:
    """Sliding-window decode: the query at position i = context_lens[b] - 1
    attends to positions max(0, i - window) .. i ("KV Cache Explained Like
    You're an LLM Engineer", section "Sliding Window Attention": token i
    attends to tokens [i - W, i], so the cache it needs is O(W)). Blocks that
    lie wholly before the window are never read (their table entries may be
    -1). q [B][H][D]; returns fp64 [B][H][D]; a context <= 0 gives zeros.
    """
    q = np.asarray(q)
    B, H, D = q.shape
    Hk = np.asarray(k_pool).shape[1]
    bs = np.asarray(k_pool).shape[2]
    g = H // Hk
    out = np.zeros((B, H, D), dtype=np.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n <= 0:
            continue
        lo = max(0, n - 1 - int(window))
        rows_k, rows_v = [], []
        for t in range(lo, n):
            blk = int(block_tables[b][t // bs])
            rows_k.append(np.asarray(k_pool)[blk, :, t % bs, :])
            rows_v.append(np.asarray(v_pool)[blk, :, t % bs, :])
        kc = _as_f64(np.stack(rows_k))
        vc = _as_f64(np.stack(rows_v))
        for h in range(H):
            out[b, h] = attend(q[b, h], kc[:, h // g, :], vc[:, h // g, :], scale)
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, context_lens, q_start_loc, scale,
                  rows=None) -> np.ndarray:
    """Causal attention of a chunk of new queries over the paged cache.

    Sequence s owns query rows q_start_loc[s] .. q_start_loc[s+1]-1; its chunk
    of L = q_start_loc[s+1] - q_start_loc[s] tokens occupies the last L
    positions of its context_lens[s] cached tokens, so query row i (0-based
    within the chunk) sits at absolute position p = context_lens[s] - L + i
    and attends to positions 0..p. q [Tq][H][D] -> fp64 out [Tq][H][D].
    ``rows`` optionally restricts the work to a list of (row, head) pairs;
    other entries are left as NaN.
    """
    q = np.asarray(q)
    Tq, H, D = q.shape
    Hk = np.asarray(k_pool).shape[1]
    g = H // Hk
    out = np.full((Tq, H, D), np.nan if rows is not None else 0.0, dtype=np.float64)
    n_seqs = len(q_start_loc) - 1
    want = None
    if rows is not None:
        want = {}
        for r, h in rows:
            want.setdefault(int(r), []).append(int(h))
    for s in range(n_seqs):
        r0, r1 = int(q_start_loc[s]), int(q_start_loc[s + 1])
        L = r1 - r0
        if L == 0:
            continue
        n = int(context_lens[s])
        if want is not None and not any(r in want for r in range(r0, r1)):
            continue
        kc = _as_f64(gather_kv(k_pool, block_tables[s], n))
        vc = _as_f64(gather_kv(v_pool, block_tables[s], n))
        for i in range(L):
            r = r0 + i
            heads = range(H) if want is None else want.get(r, [])
            p = n - L + i
            for h in heads:
                kh = h // g
                out[r, h] = attend(q[r, h], kc[:p + 1, kh, :], vc[:p + 1, kh, :], scale)
    return out
