"""Seeded synthetic workloads shaped like the pages' paged-KV examples.

Draw order for every case (one ``numpy.random.default_rng(seed)`` stream):
context lengths -> physical block placement (a random permutation of the pool)
-> q -> K -> V (token-major, one sequence after another) -> anything extra
(copy-on-write choice, divergent tokens).

Layouts (all C-contiguous):
  k_pool, v_pool  uint16 (bf16 bits) [num_blocks][n_kv_heads][block_size][head_dim]
  block tables    int32 [n_seqs][max_blocks_per_seq], unused entries = -1
  context_lens    int32 [n_seqs], counts every valid token incl. this step's
  q (decode)      uint16 [n_seqs][n_heads][head_dim]
  q (prefill)     uint16 [n_chunk_tokens][n_heads][head_dim]
  new_k, new_v    uint16 [n_new][n_kv_heads][head_dim]; slot_mapping int64 [n_new]

A slot is ``physical_block * block_size + offset``; tokens of this step
(``n_new`` per sequence) are NOT in the pool: their slots hold the fill value
and their K/V rows are returned in ``new_k``/``new_v`` for the cache-write
kernel. The fill value is bf16 NaN for parity runs (a read of an unwritten
slot then poisons the result) and 0 for timing runs.

This module holds no attention arithmetic; the only index arithmetic is the
placement of drawn rows at their slots, which is how the inputs are encoded.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = 0x7FC0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


@dataclass
class Workload:
    name: str
    seed: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    num_blocks: int
    scale: float
    block_size: int = BLOCK_SIZE
    k_pool: Optional[np.ndarray] = None
    v_pool: Optional[np.ndarray] = None
    # decode batch
    dec_tables: Optional[np.ndarray] = None
    dec_ctx: Optional[np.ndarray] = None
    q: Optional[np.ndarray] = None
    # prefill batch (chunk queries)
    pf_tables: Optional[np.ndarray] = None
    pf_ctx: Optional[np.ndarray] = None
    q_start_loc: Optional[np.ndarray] = None
    q_pf: Optional[np.ndarray] = None
    # this step's new tokens (decode tokens first, then prefill chunk tokens)
    new_k: Optional[np.ndarray] = None
    new_v: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None
    # copy-on-write (shared-prefix case)
    copy_pairs: Optional[np.ndarray] = None
    cow_seqs: Optional[np.ndarray] = None
    dec_tables_after_cow: Optional[np.ndarray] = None
    div_k: Optional[np.ndarray] = None
    div_v: Optional[np.ndarray] = None
    div_slots: Optional[np.ndarray] = None
    # logical (contiguous) per-sequence K/V, kept for small cases only
    seq_k: Optional[List[np.ndarray]] = None
    seq_v: Optional[List[np.ndarray]] = None
    meta: Dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    def kv_bytes_per_token(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim * 2


def _tables_from_placement(n_blocks_per_seq: Sequence[int], placement: np.ndarray,
                           prefix_ids: Sequence[int] = ()) -> np.ndarray:
    max_blocks = max(n_blocks_per_seq) if len(n_blocks_per_seq) else 0
    tables = np.full((len(n_blocks_per_seq), max(max_blocks, 1)), -1, dtype=np.int32)
    cursor = 0
    npre = len(prefix_ids)
    for b, nb in enumerate(n_blocks_per_seq):
        tables[b, :npre] = prefix_ids
        priv = nb - npre
        tables[b, npre:nb] = placement[cursor:cursor + priv]
        cursor += priv
    return tables


def _place(pool: np.ndarray, table_row: np.ndarray, rows: np.ndarray, start_pos: int) -> None:
    """Write rows [n][Hk][D] at logical positions start_pos.. of one sequence."""
    bs = pool.shape[2]
    n = rows.shape[0]
    pos = start_pos
    i = 0
    while i < n:
        blk = int(table_row[pos // bs])
        off = pos % bs
        take = min(bs - off, n - i)
        pool[blk, :, off:off + take, :] = rows[i:i + take].transpose(1, 0, 2)
        i += take
        pos += take


def _slots(table_row: np.ndarray, positions: Sequence[int], bs: int) -> List[int]:
    return [int(table_row[p // bs]) * bs + p % bs for p in positions]


def make_decode_case(seed: int, context_lens: Sequence[int], n_heads: int, n_kv_heads: int,
                     head_dim: int, num_blocks: Optional[int] = None, pool_factor: float = 1.25,
                     n_new: int = 0, prefix_tokens: int = 0, fill: str = "nan",
                     keep_logical: bool = True, scale: Optional[float] = None,
                     name: str = "decode", rng: Optional[np.random.Generator] = None,
                     ctx_drawn: bool = False) -> Workload:
    """A decode batch over a randomly placed paged cache.

    ``context_lens`` counts all tokens incl. the ``n_new`` of this step.
    ``prefix_tokens`` (a multiple of the block size) are shared by every
    sequence through the same physical blocks.
    """
    bs = BLOCK_SIZE
    rng = rng if rng is not None else np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    B = len(ctx)
    assert prefix_tokens % bs == 0
    npre = prefix_tokens // bs
    assert all(c >= prefix_tokens for c in ctx) or prefix_tokens == 0
    assert all(c >= n_new for c in ctx), "every context must hold its new tokens"
    nb = [max(int(math.ceil(c / bs)), npre) for c in ctx]
    needed = npre + sum(n - npre for n in nb)
    if num_blocks is None:
        num_blocks = max(int(math.ceil(pool_factor * needed)), needed)
    assert num_blocks >= needed
    perm = rng.permutation(num_blocks).astype(np.int32)
    prefix_ids = perm[:npre]
    tables = _tables_from_placement(nb, perm[npre:needed], prefix_ids)
    H, Hk, D = n_heads, n_kv_heads, head_dim
    q = _normal_bf16(rng, (B, H, D))
    fillv = BF16_NAN if fill == "nan" else 0
    k_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    v_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    new_k = np.empty((B * n_new, Hk, D), dtype=np.uint16)
    new_v = np.empty((B * n_new, Hk, D), dtype=np.uint16)
    slots = np.empty((B * n_new,), dtype=np.int64)
    seq_k: List[np.ndarray] = []
    seq_v: List[np.ndarray] = []
    for which, pool, new in (("k", k_pool, new_k), ("v", v_pool, new_v)):
        pre = _normal_bf16(rng, (prefix_tokens, Hk, D)) if prefix_tokens else None
        if pre is not None:
            _place(pool, tables[0], pre, 0)
        for b in range(B):
            c = int(ctx[b])
            priv = _normal_bf16(rng, (c - prefix_tokens, Hk, D))
            full = priv if pre is None else np.concatenate([pre, priv], axis=0)
            n_old = c - n_new
            if n_old > prefix_tokens:
                _place(pool, tables[b], full[prefix_tokens:n_old], prefix_tokens)
            if n_new:
                new[b * n_new:(b + 1) * n_new] = full[n_old:c]
            if keep_logical:
                (seq_k if which == "k" else seq_v).append(full)
    for b in range(B):
        c = int(ctx[b])
        if n_new:
            slots[b * n_new:(b + 1) * n_new] = _slots(tables[b], range(c - n_new, c), bs)
    wl = Workload(name=name, seed=seed, n_heads=H, n_kv_heads=Hk, head_dim=D,
                  num_blocks=num_blocks,
                  scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                  k_pool=k_pool, v_pool=v_pool, dec_tables=tables, dec_ctx=ctx, q=q,
                  new_k=new_k, new_v=new_v, slot_mapping=slots,
                  seq_k=seq_k if keep_logical else None,
                  seq_v=seq_v if keep_logical else None)
    wl.meta.update(needed_blocks=needed, perm_tail=perm[needed:], prefix_ids=prefix_ids,
                   n_new=n_new, prefix_tokens=prefix_tokens)
    return wl


def make_prefill_case(seed: int, chunk_ctx: Sequence[int], chunk_lens: Sequence[int],
                      decode_ctx: Sequence[int], n_heads: int, n_kv_heads: int, head_dim: int,
                      pool_factor: float = 1.25, fill: str = "nan", keep_logical: bool = True,
                      scale: Optional[float] = None, name: str = "mixed",
                      rng: Optional[np.random.Generator] = None) -> Workload:
    """Chunked-prefill sequences plus decode sequences sharing one pool.

    ``chunk_ctx[i]`` is sequence i's total length after its chunk of
    ``chunk_lens[i]`` new tokens (so the chunk starts at chunk_ctx - chunk_len).
    Every decode sequence appends one new token. New tokens are ordered decode
    tokens first, then the chunks' tokens.
    """
    bs = BLOCK_SIZE
    rng = rng if rng is not None else np.random.default_rng(seed)
    pctx = np.asarray(chunk_ctx, dtype=np.int32)
    plen = np.asarray(chunk_lens, dtype=np.int32)
    dctx = np.asarray(decode_ctx, dtype=np.int32)
    nb_p = [int(math.ceil(c / bs)) for c in pctx]
    nb_d = [int(math.ceil(c / bs)) for c in dctx]
    needed = sum(nb_p) + sum(nb_d)
    num_blocks = max(int(math.ceil(pool_factor * needed)), needed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    pf_tables = _tables_from_placement(nb_p, perm[:sum(nb_p)])
    dec_tables = _tables_from_placement(nb_d, perm[sum(nb_p):needed])
    H, Hk, D = n_heads, n_kv_heads, head_dim
    n_chunk = int(plen.sum())
    q_pf = _normal_bf16(rng, (n_chunk, H, D))
    q = _normal_bf16(rng, (len(dctx), H, D))
    fillv = BF16_NAN if fill == "nan" else 0
    k_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    v_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    n_new = len(dctx) + n_chunk
    new_k = np.empty((n_new, Hk, D), dtype=np.uint16)
    new_v = np.empty((n_new, Hk, D), dtype=np.uint16)
    slots = np.empty((n_new,), dtype=np.int64)
    seq_k: List[np.ndarray] = []
    seq_v: List[np.ndarray] = []
    for which, pool, new in (("k", k_pool, new_k), ("v", v_pool, new_v)):
        for i in range(len(pctx)):           # prefill sequences first
            c, L = int(pctx[i]), int(plen[i])
            full = _normal_bf16(rng, (c, Hk, D))
            _place(pool, pf_tables[i], full[:c - L], 0)
            off = len(dctx) + int(plen[:i].sum())
            new[off:off + L] = full[c - L:c]
            if keep_logical:
                (seq_k if which == "k" else seq_v).append(full)
        for b in range(len(dctx)):
            c = int(dctx[b])
            full = _normal_bf16(rng, (c, Hk, D))
            _place(pool, dec_tables[b], full[:c - 1], 0)
            new[b] = full[c - 1]
            if keep_logical:
                (seq_k if which == "k" else seq_v).append(full)
    for b in range(len(dctx)):
        c = int(dctx[b])
        slots[b] = _slots(dec_tables[b], [c - 1], bs)[0]
    for i in range(len(pctx)):
        c, L = int(pctx[i]), int(plen[i])
        off = len(dctx) + int(plen[:i].sum())
        slots[off:off + L] = _slots(pf_tables[i], range(c - L, c), bs)
    qsl = np.zeros(len(pctx) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(plen)
    wl = Workload(name=name, seed=seed, n_heads=H, n_kv_heads=Hk, head_dim=D,
                  num_blocks=num_blocks,
                  scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                  k_pool=k_pool, v_pool=v_pool, dec_tables=dec_tables, dec_ctx=dctx, q=q,
                  pf_tables=pf_tables, pf_ctx=pctx, q_start_loc=qsl, q_pf=q_pf,
                  new_k=new_k, new_v=new_v, slot_mapping=slots,
                  seq_k=seq_k if keep_logical else None,
                  seq_v=seq_v if keep_logical else None)
    wl.meta.update(needed_blocks=needed, n_decode_new=len(dctx), chunk_lens=plen)
    return wl


# --------------------------------------------------------------------------
# Sliding window: only blocks that reach into the window are held
# --------------------------------------------------------------------------

def make_decode_case_window(seed: int, context_lens: Sequence[int], n_heads: int, n_kv_heads: int,
                            head_dim: int, window: int, pool_factor: float = 1.25, n_new: int = 1,
                            fill: str = "nan", scale: Optional[float] = None, name: str = "decode_window",
                            rng: Optional[np.random.Generator] = None) -> Workload:
    """A decode batch whose sequences hold only the blocks that reach into the
    window of the query at position ctx - 1 (positions ctx-1-window .. ctx-1):
    table entries of blocks wholly before it are -1 (released). The first
    held block is drawn whole, so every held slot has a value.

    Draw order: context lengths -> placement -> q -> K -> V (held positions
    only, one sequence after another; this step's new token last).
    """
    bs = BLOCK_SIZE
    rng = rng if rng is not None else np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    B = len(ctx)
    assert all(c >= n_new for c in ctx)
    first_blk = [max(0, int(c) - 1 - window) // bs for c in ctx]
    nb = [int(math.ceil(c / bs)) for c in ctx]
    held = [n - f for n, f in zip(nb, first_blk)]
    needed = sum(held)
    num_blocks = max(int(math.ceil(pool_factor * needed)), needed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((B, max(nb)), -1, dtype=np.int32)
    cur = 0
    for b in range(B):
        tables[b, first_blk[b]:nb[b]] = perm[cur:cur + held[b]]
        cur += held[b]
    H, Hk, D = n_heads, n_kv_heads, head_dim
    q = _normal_bf16(rng, (B, H, D))
    fillv = BF16_NAN if fill == "nan" else 0
    k_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    v_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint16)
    new_k = np.empty((B * n_new, Hk, D), dtype=np.uint16)
    new_v = np.empty((B * n_new, Hk, D), dtype=np.uint16)
    for pool, new in ((k_pool, new_k), (v_pool, new_v)):
        for b in range(B):
            c, p0 = int(ctx[b]), first_blk[b] * bs
            rows = _normal_bf16(rng, (c - p0, Hk, D))
            if c - n_new > p0:
                _place(pool, tables[b], rows[:c - n_new - p0], p0)
            new[b * n_new:(b + 1) * n_new] = rows[c - n_new - p0:]
    slots = np.empty((B * n_new,), dtype=np.int64)
    for b in range(B):
        c = int(ctx[b])
        slots[b * n_new:(b + 1) * n_new] = _slots(tables[b], range(c - n_new, c), bs)
    wl = Workload(name=name, seed=seed, n_heads=H, n_kv_heads=Hk, head_dim=D, num_blocks=num_blocks,
                  scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                  k_pool=k_pool, v_pool=v_pool, dec_tables=tables, dec_ctx=ctx, q=q,
                  new_k=new_k, new_v=new_v, slot_mapping=slots)
    wl.meta.update(needed_blocks=needed, n_new=n_new, window=int(window))
    return wl


# --------------------------------------------------------------------------
# fp8 (E4M3) KV cache
# --------------------------------------------------------------------------

E4M3_NAN = 0x7F
_E4M3_FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def _e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Cached K/V drawn directly as E4M3 codes: uniform over the 254 finite
    bit patterns (both signs, zeros, subnormals, up to the largest finite
    value). No rounding is involved: the codes are the input."""
    return _E4M3_FINITE[rng.integers(0, len(_E4M3_FINITE), size=shape)]


def make_decode_case_fp8(seed: int, context_lens: Sequence[int], n_heads: int, n_kv_heads: int,
                         head_dim: int, num_blocks: Optional[int] = None, pool_factor: float = 1.25,
                         n_new: int = 1, fill: str = "nan", scale: Optional[float] = None,
                         name: str = "decode_fp8", rng: Optional[np.random.Generator] = None
                         ) -> Workload:
    """A decode batch over a randomly placed paged cache of E4M3 codes.

    Draw order: context lengths -> placement -> q -> cached K codes -> cached
    V codes (one sequence after another) -> this step's new K -> new V (bf16,
    N(0,1); the cache write quantises them) -> per-KV-head scales for K and
    for V, each 2^-6 * (1 + u), u ~ U[0, 1), as fp32.

    Layouts: k_pool, v_pool uint8 [num_blocks][n_kv_heads][block_size][head_dim]
    (fill: E4M3 NaN 0x7F for parity runs, 0 for timing runs); k_scale, v_scale
    float32 [n_kv_heads]; q, new_k, new_v bf16 bits as in ``make_decode_case``.
    """
    bs = BLOCK_SIZE
    rng = rng if rng is not None else np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    B = len(ctx)
    assert all(c >= n_new for c in ctx), "every context must hold its new tokens"
    nb = [int(math.ceil(c / bs)) for c in ctx]
    needed = sum(nb)
    if num_blocks is None:
        num_blocks = max(int(math.ceil(pool_factor * needed)), needed)
    assert num_blocks >= needed
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_placement(nb, perm[:needed])
    H, Hk, D = n_heads, n_kv_heads, head_dim
    q = _normal_bf16(rng, (B, H, D))
    fillv = E4M3_NAN if fill == "nan" else 0
    k_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint8)
    v_pool = np.full((num_blocks, Hk, bs, D), fillv, dtype=np.uint8)
    for pool in (k_pool, v_pool):
        for b in range(B):
            n_old = int(ctx[b]) - n_new
            if n_old > 0:
                _place(pool, tables[b], _e4m3_codes(rng, (n_old, Hk, D)), 0)
    new_k = _normal_bf16(rng, (B * n_new, Hk, D))
    new_v = _normal_bf16(rng, (B * n_new, Hk, D))
    slots = np.empty((B * n_new,), dtype=np.int64)
    for b in range(B):
        c = int(ctx[b])
        if n_new:
            slots[b * n_new:(b + 1) * n_new] = _slots(tables[b], range(c - n_new, c), bs)
    k_scale = (2.0 ** -6 * (1.0 + rng.random(Hk))).astype(np.float32)
    v_scale = (2.0 ** -6 * (1.0 + rng.random(Hk))).astype(np.float32)
    wl = Workload(name=name, seed=seed, n_heads=H, n_kv_heads=Hk, head_dim=D,
                  num_blocks=num_blocks,
                  scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                  k_pool=k_pool, v_pool=v_pool, dec_tables=tables, dec_ctx=ctx, q=q,
                  new_k=new_k, new_v=new_v, slot_mapping=slots)
    wl.meta.update(needed_blocks=needed, n_new=n_new, kv_dtype="fp8_e4m3",
                   k_scale=k_scale, v_scale=v_scale)
    return wl


# --------------------------------------------------------------------------
# The named workloads. Seed = workload index (0..4); the fp8 variant of the
# 8B batch reuses the 8B batch's seed so its context lengths match.
# --------------------------------------------------------------------------

def _tiny_mha(fill="nan", keep_logical=True):
    """4 sequences, context {1,15,16,37}, 4 q = 4 kv heads, head_dim 64, pool 32."""
    return make_decode_case(0, [1, 15, 16, 37], 4, 4, 64, num_blocks=32, n_new=0,
                            fill=fill, keep_logical=keep_logical, scale=1.0 / 8.0,
                            name="tiny_mha_b4_d64")


def _mha_7b(fill="nan", keep_logical=False):
    """Llama-7B-class MHA layer: batch 8 x context 2048, 32 heads, d 128, pool 4096."""
    return make_decode_case(1, [2048] * 8, 32, 32, 128, num_blocks=4096, n_new=1,
                            fill=fill, keep_logical=keep_logical, name="mha7b_b8_ctx2048")


def _gqa_8b(fill="nan", keep_logical=False):
    """Llama-3-8B-shaped GQA: batch 64, context U{128..4096}, 32 q / 8 kv heads."""
    rng = np.random.default_rng(2)
    ctx = rng.integers(128, 4096, size=64, endpoint=True)
    return make_decode_case(2, ctx, 32, 8, 128, pool_factor=1.25, n_new=1, fill=fill,
                            keep_logical=keep_logical, name="gqa8b_b64_ctx128-4096", rng=rng)


def _gqa_70b_cow(fill="nan", keep_logical=False):
    """70B-shaped GQA: 100 sequences x 4096, 512-token shared prefix (32 blocks,
    refcount 100), 64 q / 8 kv heads; 10 sequences copy-on-write the last
    shared block and write one divergent token into their private copy."""
    rng = np.random.default_rng(3)
    B, pre, ctx = 100, 512, 4096
    npre = pre // BLOCK_SIZE
    needed = npre + B * (ctx // BLOCK_SIZE - npre)
    num_blocks = needed + 10
    wl = make_decode_case(3, [ctx] * B, 64, 8, 128, num_blocks=num_blocks, n_new=1,
                          prefix_tokens=pre, fill=fill, keep_logical=keep_logical,
                          name="gqa70b_b100_ctx4096_prefix512_cow", rng=rng)
    cow = np.sort(rng.choice(B, size=10, replace=False)).astype(np.int32)
    dst = wl.meta["perm_tail"][:10]
    src = int(wl.dec_tables[0, npre - 1])
    wl.copy_pairs = np.array([[src, int(d)] for d in dst], dtype=np.int64)
    t2 = wl.dec_tables.copy()
    t2[cow, npre - 1] = dst
    wl.dec_tables_after_cow = t2
    wl.cow_seqs = cow
    wl.div_k = _normal_bf16(rng, (10, wl.n_kv_heads, wl.head_dim))
    wl.div_v = _normal_bf16(rng, (10, wl.n_kv_heads, wl.head_dim))
    # the divergent token overwrites the last slot of the private copy
    wl.div_slots = (dst.astype(np.int64) * BLOCK_SIZE + (BLOCK_SIZE - 1)).astype(np.int64)
    return wl


def _mixed(fill="nan", keep_logical=False):
    """4 sequences at 32768 receiving a 512-token causal chunk + 60 decode
    sequences with context U{256..8192}; 32 q / 8 kv heads, d 128."""
    rng = np.random.default_rng(4)
    dctx = rng.integers(256, 8192, size=60, endpoint=True)
    return make_prefill_case(4, [32768] * 4, [512] * 4, dctx, 32, 8, 128, fill=fill,
                             keep_logical=keep_logical, name="mixed_prefill4x512_at32k_decode60",
                             rng=rng)


def _gqa_8b_fp8(fill="nan", keep_logical=False):
    """The 8B-shaped GQA batch (same context lengths as ``gqa_8b``) over an
    E4M3 cache with per-KV-head scales."""
    rng = np.random.default_rng(2)
    ctx = rng.integers(128, 4096, size=64, endpoint=True)
    return make_decode_case_fp8(2, ctx, 32, 8, 128, pool_factor=1.25, n_new=1, fill=fill,
                                name="gqa8b_fp8_b64_ctx128-4096", rng=rng)


def _swa_mistral(fill="nan", keep_logical=False):
    """Mistral-7B-shaped sliding-window decode: 32 sequences, context
    U{4096..32768}, window 4096, 32 q / 8 kv heads, d 128; only the blocks
    that reach into each window are held."""
    rng = np.random.default_rng(5)
    ctx = rng.integers(4096, 32768, size=32, endpoint=True)
    return make_decode_case_window(5, ctx, 32, 8, 128, 4096, fill=fill,
                                   name="swa_mistral_b32_ctx4k-32k_w4096", rng=rng)


WORKLOADS = {
    "tiny_mha": _tiny_mha,
    "mha_7b": _mha_7b,
    "gqa_8b": _gqa_8b,
    "gqa_70b_cow": _gqa_70b_cow,
    "mixed": _mixed,
    "gqa_8b_fp8": _gqa_8b_fp8,
    "swa_mistral": _swa_mistral,
}


def make_workload(name: str, fill: str = "nan", keep_logical: Optional[bool] = None) -> Workload:
    fn = WORKLOADS[name]
    if keep_logical is None:
        return fn(fill=fill)
    return fn(fill=fill, keep_logical=keep_logical)
