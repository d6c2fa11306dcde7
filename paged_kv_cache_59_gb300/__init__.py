"""Python binding of libpagedkv.so: PagedAttention decode over a paged bf16 KV
cache on GB300, the cache-write and block-copy kernels, chunked prefill, and
the host block manager.

Argument marshalling only: each function reads sizes from tensor shapes,
checks device, dtype and contiguity, and calls the C entry point of the same
name on the current CUDA stream. Every computation runs in the library's
CUDA kernels; a missing library or a CPU tensor is an error.

Tensors: bf16 tensors may be torch.bfloat16 or int16/uint16 carrying bf16
bits. Pools are [num_blocks][n_kv_heads][16][head_dim]; block tables int32
[n_seqs][max_blocks]; context lengths int32 [n_seqs]; slots int64.
"""
from __future__ import annotations

import ctypes as C
from typing import List, Optional, Sequence, Tuple

from . import _capi
from ._capi import PagedKVError, check, load  # noqa: F401

__all__ = [
    "pa_decode", "pa_decode_tc", "pa_decode_workspace_bytes", "pa_decode_partition_tokens", "decode_workspace", "pa_decode_noalloc", "pa_reshape_and_cache",
    "pa_copy_blocks", "pa_prefill_paged", "pa_prefill_paged_ex", "pa_prefill_workspace_bytes",
    "prefill_workspace", "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_decode_window",
    "pa_swap_out_blocks", "pa_swap_in_blocks", "pa_get_device_error",
    "BlockManager", "load", "PagedKVError",
]


def _torch():
    import torch
    return torch


_BF16_LIKE = None


def _ptr(t, what: str, bf16: bool = False, dtype=None):
    torch = _torch()
    global _BF16_LIKE
    if _BF16_LIKE is None:
        _BF16_LIKE = {torch.bfloat16, torch.int16, getattr(torch, "uint16", torch.int16)}
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{what} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if bf16 and t.dtype not in _BF16_LIKE:
        raise TypeError(f"{what} must hold bf16 (bfloat16 or 16-bit integer bits), got {t.dtype}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def pa_decode_workspace_bytes(n_seqs: int, n_heads: int, head_dim: int, max_context_len: int,
                              partition_tokens: int = 0) -> int:
    return int(load().pa_decode_workspace_bytes(n_seqs, n_heads, head_dim, max_context_len,
                                                partition_tokens))


def pa_decode_partition_tokens(n_seqs: int, n_heads: int, n_kv_heads: int, head_dim: int,
                               max_context_len: int, window: int = -1, elem_bytes: int = 2) -> int:
    """The partition size the decode entry points use with partition_tokens=0."""
    st = int(load().pa_decode_partition_tokens(n_seqs, n_heads, n_kv_heads, head_dim, max_context_len,
                                               window, elem_bytes))
    check("pa_decode_partition_tokens", min(st, 0))
    return st


def decode_workspace(q, max_context_len: int, partition_tokens: int = 0):
    """A workspace tensor sized for pa_decode on this q shape and context bound."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    nbytes = pa_decode_workspace_bytes(n_seqs, n_heads, head_dim, max_context_len, partition_tokens)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)


def pa_decode(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
              max_context_len: int, workspace=None, partition_tokens: int = 0, stream=None,
              tensor_cores: bool = False) -> None:
    """out[b][h] = softmax(scale * q[b][h] . K_b^T) V_b over each sequence's
    paged K/V. q, out: [n_seqs][n_heads][head_dim]. tensor_cores=True calls
    pa_decode_tc (the warp-level MMA kernel at every group size)."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    if hd2 != head_dim or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != n_seqs or context_lens.numel() != n_seqs:
        raise ValueError("block_tables must be [n_seqs][max_blocks], context_lens [n_seqs]")
    ws_ptr, ws_bytes = C.c_void_p(None), 0
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    lib = load()
    st = (lib.pa_decode_tc if tensor_cores else lib.pa_decode_ex)(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_context_len), num_blocks,
        int(partition_tokens), ws_ptr, ws_bytes, _stream(stream))
    check("pa_decode_tc" if tensor_cores else "pa_decode", st)


def pa_decode_tc(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                 max_context_len: int, workspace=None, partition_tokens: int = 0, stream=None) -> None:
    """pa_decode on the tensor-core (warp-level MMA) partition kernel, any group size."""
    pa_decode(out, q, k_pool, v_pool, block_tables, context_lens, scale, max_context_len, workspace,
              partition_tokens, stream, tensor_cores=True)


def pa_decode_noalloc(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                      max_context_len: int, stream=None) -> None:
    """pa_decode without a caller workspace, for callers that cannot allocate
    device memory: the split-K scratch is a fixed 32 MiB array inside the
    library shared by all calls on a device (calls that overlap on the GPU
    race on it). Batches needing more scratch raise (PA_ERR_WORKSPACE)."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    if hd2 != head_dim or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != n_seqs or context_lens.numel() != n_seqs:
        raise ValueError("block_tables must be [n_seqs][max_blocks], context_lens [n_seqs]")
    st = load().pa_decode_noalloc(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_context_len), num_blocks,
        _stream(stream))
    check("pa_decode_noalloc", st)


def pa_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, stream=None) -> None:
    """Writes k[t], v[t] ([n_tokens][n_kv_heads][head_dim]) to slot_mapping[t]."""
    torch = _torch()
    n_tokens, n_kv_heads, head_dim = k.shape
    num_blocks, hk2, block_size, hd2 = k_pool.shape
    if (hk2, hd2) != (n_kv_heads, head_dim) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between k/v and the pools")
    if slot_mapping.numel() != n_tokens:
        raise ValueError("slot_mapping must have n_tokens entries")
    st = load().pa_reshape_and_cache(
        _ptr(k, "k", bf16=True), _ptr(v, "v", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(slot_mapping, "slot_mapping", dtype=torch.int64),
        n_tokens, n_kv_heads, head_dim, block_size, num_blocks, _stream(stream))
    check("pa_reshape_and_cache", st)


def _fp8_pool(t, what: str):
    torch = _torch()
    if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise TypeError(f"{what} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    return _ptr(t, what)


def pa_decode_window(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                     max_context_len: int, window: int, workspace=None, partition_tokens: int = 0,
                     stream=None) -> None:
    """Sliding-window decode: the query at position ctx-1 attends to positions
    ctx-1-window .. ctx-1; blocks wholly before that are never read."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    if hd2 != head_dim or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != n_seqs or context_lens.numel() != n_seqs:
        raise ValueError("block_tables must be [n_seqs][max_blocks], context_lens [n_seqs]")
    ws_ptr, ws_bytes = C.c_void_p(None), 0
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    st = load().pa_decode_window(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_context_len), num_blocks, int(window),
        int(partition_tokens), ws_ptr, ws_bytes, _stream(stream))
    check("pa_decode_window", st)


def _host_pinned(t, what: str):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{what} must be page-locked host memory (pin_memory=True)")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _swap_args(k_pool, host_k, host_v, block_ids):
    torch = _torch()
    num_blocks, n_kv_heads, block_size, head_dim = k_pool.shape
    eb = k_pool.element_size()
    n = block_ids.numel()
    need = n * n_kv_heads * block_size * head_dim * eb
    for h, name in ((host_k, "host_k"), (host_v, "host_v")):
        if h.numel() * h.element_size() < need:
            raise ValueError(f"{name} holds fewer than {need} bytes")
    return (n, n_kv_heads, head_dim, block_size, eb, num_blocks,
            _ptr(block_ids, "block_ids", dtype=torch.int32) if n else C.c_void_p(None))


def pa_swap_out_blocks(k_pool, v_pool, block_ids, host_k, host_v, stream=None) -> None:
    """host_k[i], host_v[i] := pool block block_ids[i] (K and V, all heads);
    host buffers page-locked, block_ids int32 on the device."""
    n, hk, d, bs, eb, nb, ids = _swap_args(k_pool, host_k, host_v, block_ids)
    st = load().pa_swap_out_blocks(_ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"), ids, n,
                                   _host_pinned(host_k, "host_k"), _host_pinned(host_v, "host_v"), hk, d, bs,
                                   eb, nb, _stream(stream))
    check("pa_swap_out_blocks", st)


def pa_swap_in_blocks(host_k, host_v, k_pool, v_pool, block_ids, stream=None) -> None:
    """pool block block_ids[i] := host_k[i], host_v[i]."""
    n, hk, d, bs, eb, nb, ids = _swap_args(k_pool, host_k, host_v, block_ids)
    st = load().pa_swap_in_blocks(_host_pinned(host_k, "host_k"), _host_pinned(host_v, "host_v"),
                                  _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"), ids, n, hk, d, bs, eb, nb,
                                  _stream(stream))
    check("pa_swap_in_blocks", st)


def pa_reshape_and_cache_fp8(k, v, k_pool, v_pool, slot_mapping, k_scale, v_scale, stream=None) -> None:
    """Encodes k[t], v[t] (bf16 [n_tokens][n_kv_heads][head_dim]) as E4M3 codes
    of x / scale[head] into the uint8 pools at slot_mapping[t]."""
    torch = _torch()
    n_tokens, n_kv_heads, head_dim = k.shape
    num_blocks, hk2, block_size, hd2 = k_pool.shape
    if (hk2, hd2) != (n_kv_heads, head_dim) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between k/v and the pools")
    if slot_mapping.numel() != n_tokens or k_scale.numel() != n_kv_heads or v_scale.numel() != n_kv_heads:
        raise ValueError("slot_mapping needs n_tokens entries, k_scale/v_scale n_kv_heads")
    st = load().pa_reshape_and_cache_fp8(
        _ptr(k, "k", bf16=True), _ptr(v, "v", bf16=True), _fp8_pool(k_pool, "k_pool"),
        _fp8_pool(v_pool, "v_pool"), _ptr(slot_mapping, "slot_mapping", dtype=torch.int64),
        _ptr(k_scale, "k_scale", dtype=torch.float32), _ptr(v_scale, "v_scale", dtype=torch.float32),
        n_tokens, n_kv_heads, head_dim, block_size, num_blocks, _stream(stream))
    check("pa_reshape_and_cache_fp8", st)


def pa_decode_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale: float,
                  max_context_len: int, workspace=None, partition_tokens: int = 0, stream=None) -> None:
    """pa_decode over an E4M3 cache: K and V are decode(code) * scale of their
    KV head. Pools uint8 [num_blocks][n_kv_heads][16][head_dim]."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    if hd2 != head_dim or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != n_seqs or context_lens.numel() != n_seqs:
        raise ValueError("block_tables must be [n_seqs][max_blocks], context_lens [n_seqs]")
    if k_scale.numel() != n_kv_heads or v_scale.numel() != n_kv_heads:
        raise ValueError("k_scale and v_scale need one entry per KV head")
    ws_ptr, ws_bytes = C.c_void_p(None), 0
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    st = load().pa_decode_fp8(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _fp8_pool(k_pool, "k_pool"),
        _fp8_pool(v_pool, "v_pool"), _ptr(k_scale, "k_scale", dtype=torch.float32),
        _ptr(v_scale, "v_scale", dtype=torch.float32), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_context_len), num_blocks,
        int(partition_tokens), ws_ptr, ws_bytes, _stream(stream))
    check("pa_decode_fp8", st)


def pa_decode_plan(context_lens, n_heads: int, n_kv_heads: int, head_dim: int, max_blocks_per_seq: int,
                   max_context_len: int, num_blocks: int, window: int = -1, elem_bytes: int = 2,
                   partition_tokens: int = 0):
    """The decode call's work items, longest partitions first, from HOST
    context lengths (a sequence of ints or an int32 array): an int32 numpy
    array [n_items][4] of (partition, kv head, sequence, 0)."""
    import numpy as np
    ctx = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32).reshape(-1))
    args = (ctx.ctypes.data_as(C.c_void_p), len(ctx), n_heads, n_kv_heads, head_dim, max_blocks_per_seq,
            int(max_context_len), num_blocks, int(window), elem_bytes, int(partition_tokens))
    n = int(load().pa_decode_plan(*args, None, 0))
    check("pa_decode_plan", min(n, 0))
    items = np.zeros((max(n, 1), 4), dtype=np.int32)
    st = int(load().pa_decode_plan(*args, items.ctypes.data_as(C.c_void_p), n))
    check("pa_decode_plan", min(st, 0))
    return items[:st]


def pa_decode_planned(out, q, k_pool, v_pool, block_tables, context_lens, scale: float, max_context_len: int,
                      items, k_scale=None, v_scale=None, window: int = -1, workspace=None,
                      partition_tokens: int = 0, stream=None) -> None:
    """pa_decode (bf16 pools), pa_decode_fp8 (uint8 pools with k_scale and
    v_scale) or, with window >= 0, pa_decode_window, run from a plan: items is
    pa_decode_plan's output for the same lengths and arguments, on the device
    (int32 [n_items][4])."""
    torch = _torch()
    n_seqs, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    if hd2 != head_dim or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.dim() != 2 or block_tables.shape[0] != n_seqs or context_lens.numel() != n_seqs:
        raise ValueError("block_tables must be [n_seqs][max_blocks], context_lens [n_seqs]")
    if items.dim() != 2 or items.shape[1] != 4:
        raise ValueError("items must be int32 [n_items][4]")
    fp8 = k_pool.dtype == torch.uint8
    if fp8 != (k_scale is not None) or (k_scale is None) != (v_scale is None):
        raise ValueError("an fp8 (uint8) pool needs k_scale and v_scale, a bf16 pool neither")
    ws_ptr, ws_bytes = C.c_void_p(None), 0
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    if fp8:
        kp, vp_ = _fp8_pool(k_pool, "k_pool"), _fp8_pool(v_pool, "v_pool")
        ks = _ptr(k_scale, "k_scale", dtype=torch.float32)
        vs = _ptr(v_scale, "v_scale", dtype=torch.float32)
    else:
        kp, vp_ = _ptr(k_pool, "k_pool", bf16=True), _ptr(v_pool, "v_pool", bf16=True)
        ks = vs = C.c_void_p(None)
    st = load().pa_decode_planned(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), kp, vp_, ks, vs,
        _ptr(block_tables, "block_tables", dtype=torch.int32), _ptr(context_lens, "context_lens", dtype=torch.int32),
        float(scale), n_heads, n_kv_heads, head_dim, block_size, n_seqs, block_tables.shape[1],
        int(max_context_len), num_blocks, int(window), int(partition_tokens),
        _ptr(items, "items", dtype=torch.int32), items.shape[0], ws_ptr, ws_bytes, _stream(stream))
    check("pa_decode_planned", st)


def pa_copy_blocks(k_pool, v_pool, block_mapping, stream=None) -> None:
    """block_mapping int64 [n][2] (src, dst) on the device: dst block := src block.
    The pools may be bf16 or fp8 (uint8 E4M3 codes); the element size is read
    from k_pool."""
    torch = _torch()
    num_blocks, n_kv_heads, block_size, head_dim = k_pool.shape
    n_pairs = block_mapping.shape[0] if block_mapping.numel() else 0
    if k_pool.dtype == torch.uint8:
        kp, vp_, eb = _fp8_pool(k_pool, "k_pool"), _fp8_pool(v_pool, "v_pool"), 1
    else:
        kp, vp_, eb = _ptr(k_pool, "k_pool", bf16=True), _ptr(v_pool, "v_pool", bf16=True), 2
    if v_pool.dtype != k_pool.dtype or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("k_pool and v_pool must have the same shape and dtype")
    st = load().pa_copy_blocks_ex(
        kp, vp_, _ptr(block_mapping, "block_mapping", dtype=torch.int64) if n_pairs else C.c_void_p(None),
        n_pairs, n_kv_heads, head_dim, block_size, eb, num_blocks, _stream(stream))
    check("pa_copy_blocks_ex", st)


def pa_prefill_paged(out, q, k_pool, v_pool, block_tables, context_lens, q_start_loc,
                     scale: float, max_chunk_len: int, stream=None) -> None:
    """Causal attention of each sequence's chunk rows over its paged cache."""
    torch = _torch()
    n_rows, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    n_seqs = context_lens.numel()
    if hd2 != head_dim or tuple(out.shape) != tuple(q.shape) or q_start_loc.numel() != n_seqs + 1:
        raise ValueError("shape mismatch in pa_prefill_paged arguments")
    st = load().pa_prefill_paged(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32),
        _ptr(q_start_loc, "q_start_loc", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_chunk_len), num_blocks,
        _stream(stream))
    check("pa_prefill_paged", st)


def pa_prefill_workspace_bytes(n_seqs: int, n_heads: int, n_kv_heads: int, max_chunk_len: int,
                               splits: int = 0) -> int:
    return int(load().pa_prefill_workspace_bytes(n_seqs, n_heads, n_kv_heads, max_chunk_len, splits))


def prefill_workspace(q, n_seqs: int, n_kv_heads: int, max_chunk_len: int, splits: int = 0):
    """A workspace tensor for pa_prefill_paged_ex (None when no split is needed)."""
    torch = _torch()
    nbytes = pa_prefill_workspace_bytes(n_seqs, q.shape[1], n_kv_heads, max_chunk_len, splits)
    return torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None


def pa_prefill_paged_ex(out, q, k_pool, v_pool, block_tables, context_lens, q_start_loc, scale: float,
                        max_chunk_len: int, splits: int = 0, workspace=None, stream=None) -> None:
    """pa_prefill_paged with each query-tile pair's key range split into pieces
    (splits = 0: chosen from the grid and the SM count) merged afterwards."""
    torch = _torch()
    n_rows, n_heads, head_dim = q.shape
    num_blocks, n_kv_heads, block_size, hd2 = k_pool.shape
    n_seqs = context_lens.numel()
    if hd2 != head_dim or tuple(out.shape) != tuple(q.shape) or q_start_loc.numel() != n_seqs + 1:
        raise ValueError("shape mismatch in pa_prefill_paged_ex arguments")
    ws_ptr, ws_bytes = C.c_void_p(None), 0
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    st = load().pa_prefill_paged_ex(
        _ptr(out, "out", bf16=True), _ptr(q, "q", bf16=True), _ptr(k_pool, "k_pool", bf16=True),
        _ptr(v_pool, "v_pool", bf16=True), _ptr(block_tables, "block_tables", dtype=torch.int32),
        _ptr(context_lens, "context_lens", dtype=torch.int32),
        _ptr(q_start_loc, "q_start_loc", dtype=torch.int32), float(scale), n_heads, n_kv_heads,
        head_dim, block_size, n_seqs, block_tables.shape[1], int(max_chunk_len), num_blocks, int(splits),
        ws_ptr, ws_bytes, _stream(stream))
    check("pa_prefill_paged_ex", st)


def pa_get_device_error() -> int:
    """Reads and clears the device error word (a PA_DEVERR_* mask)."""
    v = C.c_int(0)
    check("pa_get_device_error", load().pa_get_device_error(C.byref(v)))
    return v.value


class BlockManager:
    """Host block manager (free list, refcounts, fork, copy-on-write) in the
    library; builds block tables, slots and copy pairs."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._lib = load()
        self._h = self._lib.pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("pa_bm_create failed")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_bm_destroy(h)
            self._h = None

    def add_seq(self, seq_id: int) -> None:
        check("pa_bm_add_seq", self._lib.pa_bm_add_seq(self._h, seq_id))

    def append_tokens(self, seq_id: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        slots = (C.c_int64 * max(n, 1))()
        pairs = (C.c_int64 * 2)()
        ncow = C.c_int(0)
        check("pa_bm_append_tokens", self._lib.pa_bm_append_tokens(
            self._h, seq_id, n, slots, pairs, 1, C.byref(ncow)))
        cow = [(pairs[0], pairs[1])] if ncow.value else []
        return list(slots)[:n], cow

    def make_private(self, seq_id: int, logical_block: int) -> List[Tuple[int, int]]:
        pair = (C.c_int64 * 2)()
        n = C.c_int(0)
        check("pa_bm_make_private", self._lib.pa_bm_make_private(
            self._h, seq_id, logical_block, pair, C.byref(n)))
        return [(pair[0], pair[1])] if n.value else []

    def fork(self, parent: int, child: int) -> None:
        check("pa_bm_fork", self._lib.pa_bm_fork(self._h, parent, child))

    def free_seq(self, seq_id: int) -> None:
        check("pa_bm_free_seq", self._lib.pa_bm_free_seq(self._h, seq_id))

    def _swap(self, fn: str, seq_id: int) -> List[int]:
        n = C.c_int(0)
        st = getattr(self._lib, fn)(self._h, seq_id, None, 0, C.byref(n))
        if st == _capi.PA_OK:
            return []
        if st != _capi.PA_ERR_CAPACITY:
            check(fn, st)
        buf = (C.c_int32 * n.value)()
        check(fn, getattr(self._lib, fn)(self._h, seq_id, buf, n.value, C.byref(n)))
        return list(buf)[:n.value]

    def swap_out(self, seq_id: int) -> List[int]:
        """Releases the sequence's private tail; returns its block ids (copy
        their contents to host memory before anything reuses them)."""
        return self._swap("pa_bm_swap_out", seq_id)

    def swap_in(self, seq_id: int) -> List[int]:
        """Re-allocates a swapped sequence's tail; returns the new block ids
        (copy the contents back into them)."""
        return self._swap("pa_bm_swap_in", seq_id)

    def cache_blocks(self, seq_id: int, tokens: Sequence[int]) -> int:
        """Registers the sequence's full blocks in the prefix cache; returns
        how many entries were added."""
        arr = (C.c_int32 * max(len(tokens), 1))(*tokens)
        n = C.c_int(0)
        check("pa_bm_cache_blocks", self._lib.pa_bm_cache_blocks(self._h, seq_id, arr, len(tokens), C.byref(n)))
        return n.value

    def add_seq_cached(self, seq_id: int, tokens: Sequence[int]) -> int:
        """Starts a sequence on the longest cached prefix of tokens; returns
        the number of tokens it already holds."""
        arr = (C.c_int32 * max(len(tokens), 1))(*tokens)
        n = C.c_int64(0)
        check("pa_bm_add_seq_cached", self._lib.pa_bm_add_seq_cached(self._h, seq_id, arr, len(tokens),
                                                                      C.byref(n)))
        return n.value

    def num_cached(self) -> int:
        return self._lib.pa_bm_num_cached(self._h)

    def release_before(self, seq_id: int, first_pos: int) -> int:
        """Drops the blocks wholly before logical position first_pos (sliding
        window); their table entries become -1. Returns how many were dropped."""
        n = C.c_int(0)
        check("pa_bm_release_before", self._lib.pa_bm_release_before(self._h, seq_id, first_pos, C.byref(n)))
        return n.value

    def block_table(self, seq_id: int) -> List[int]:
        n = C.c_int(0)
        st = self._lib.pa_bm_block_table(self._h, seq_id, None, 0, C.byref(n))
        if st not in (_capi.PA_OK, _capi.PA_ERR_CAPACITY):
            check("pa_bm_block_table", st)
        buf = (C.c_int32 * max(n.value, 1))()
        check("pa_bm_block_table", self._lib.pa_bm_block_table(self._h, seq_id, buf, n.value,
                                                               C.byref(n)))
        return list(buf)[:n.value]

    def seq_len(self, seq_id: int) -> int:
        v = self._lib.pa_bm_seq_len(self._h, seq_id)
        if v < 0:
            check("pa_bm_seq_len", int(v))
        return int(v)

    def num_free(self) -> int:
        return int(self._lib.pa_bm_num_free(self._h))

    def refcount(self, block_id: int) -> int:
        v = self._lib.pa_bm_refcount(self._h, block_id)
        if v < 0:
            check("pa_bm_refcount", v)
        return int(v)

    def build_batch(self, seq_ids: Sequence[int], max_blocks: int):
        """(tables int32 [n][max_blocks], context_lens int32 [n]) as numpy arrays."""
        import numpy as np
        n = len(seq_ids)
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tabs = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty((n,), dtype=np.int32)
        check("pa_bm_build_batch", self._lib.pa_bm_build_batch(
            self._h, ids.ctypes.data_as(C.POINTER(C.c_int64)), n, max_blocks,
            tabs.ctypes.data_as(C.POINTER(C.c_int32)), lens.ctypes.data_as(C.POINTER(C.c_int32))))
        return tabs, lens
