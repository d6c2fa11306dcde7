"""GPU parity for PagedAttention decode against the fp64 oracle.

Tolerance (per element): |gpu - ref| <= 2e-3 + 1e-2 * |ref|.
Cases span several 16-token blocks and partitions with ragged tails, every
supported head_dim / GQA group, split-K partition sizes from the smallest to
one-partition, the edge contexts 0, 1, 15, 16, 17, and the full-size
workloads (all rows compared where the oracle is fast, sampled rows
otherwise).
"""
import math

import numpy as np
import pytest

from oracle.attention import paged_decode, paged_decode_rows
from oracle.cache_ops import copy_blocks as o_copy
from oracle.cache_ops import reshape_and_cache as o_rac
from tests._gpu import (assert_attention_close, bf16_to_f64, check_device_error, dev, host_bits,
                        torch_cuda)
from workloads import make_decode_case, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def gpu_decode(pk, q, kp, vp, tables, ctx, scale, max_ctx, pt=0):
    torch = torch_cuda()
    q_d = q if not isinstance(q, np.ndarray) else dev(q)
    out = torch.empty_like(q_d)
    n_seqs, H, D = q_d.shape
    ws_bytes = pk.pa_decode_workspace_bytes(n_seqs, H, D, max_ctx, pt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    pk.pa_decode(out, q_d, kp, vp, tables if not isinstance(tables, np.ndarray) else dev(tables),
                 ctx if not isinstance(ctx, np.ndarray) else dev(ctx), scale, max_ctx,
                 workspace=ws, partition_tokens=pt)
    torch.cuda.synchronize()
    return host_bits(out)


def test_tiny_workload(pk):
    wl = make_workload("tiny_mha")
    got = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                     wl.scale, int(wl.dec_ctx.max()))
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "tiny")
    # context 1: the output is v_0 exactly (one weight of 1.0)
    assert np.array_equal(got[0], wl.seq_v[0][0])
    check_device_error(0)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("pt", [0, 64, 128])
def test_shapes_groups_partitions(pk, D, H, Hk, pt):
    ctx = [1, 15, 16, 17, 37, 64, 129, 300, 513, 1000]
    wl = make_decode_case(100 + D + H + Hk + pt, ctx, H, Hk, D)
    got = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                     wl.scale, max(ctx), pt)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, f"D={D} H={H} Hk={Hk} pt={pt}")
    check_device_error(0)


@pytest.mark.parametrize("pt", [64, 512, 2048])
def test_long_context_partitions(pk, pt):
    ctx = [4096, 2049, 3000, 17]
    wl = make_decode_case(200 + pt, ctx, 32, 8, 128)
    got = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                     wl.scale, max(ctx), pt)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, f"pt={pt}")
    check_device_error(0)


@pytest.mark.parametrize("H,Hk", [(8, 2), (64, 8)])   # group 8 at head_dim 128: tensor-core kernel
def test_zero_context_rows_are_zero(pk, H, Hk):
    wl = make_decode_case(300, [0, 20, 0, 33], H, Hk, 128)
    got = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                     wl.scale, 33, 64)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "zero ctx")


@pytest.mark.parametrize("H,Hk", [(8, 2), (64, 8)])
def test_hot_logits_do_not_overflow(pk, H, Hk):
    """q scaled x20: logits of order +-100, exp without max-subtraction would overflow."""
    wl = make_decode_case(301, [77, 500, 1], H, Hk, 128)
    qf = bf16_to_f64(wl.q) * 20.0
    q_hot = ((qf.astype(np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    got = gpu_decode(pk, q_hot, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                     wl.scale, 500, 128)
    ref = paged_decode(q_hot, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "hot")


@pytest.mark.parametrize("H,Hk", [(32, 8), (64, 8)])
def test_block_permutation_gives_identical_bits(pk, H, Hk):
    wl = make_decode_case(302, [40, 300, 1000, 16], H, Hk, 128)
    a = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx,
                   wl.scale, 1000, 256)
    pi = np.random.default_rng(9).permutation(wl.num_blocks)
    kp = np.empty_like(wl.k_pool)
    vp = np.empty_like(wl.v_pool)
    kp[pi] = wl.k_pool
    vp[pi] = wl.v_pool
    tabs = np.where(wl.dec_tables >= 0, pi[np.maximum(wl.dec_tables, 0)], -1).astype(np.int32)
    b = gpu_decode(pk, wl.q, dev(kp), dev(vp), tabs, wl.dec_ctx, wl.scale, 1000, 256)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("H,Hk,D", [(4, 4, 64), (64, 8, 128)])
def test_bad_block_id_is_flagged_not_faulted(pk, H, Hk, D):
    wl = make_decode_case(303, [40, 40], H, Hk, D)
    tabs = wl.dec_tables.copy()
    tabs[1, 1] = wl.num_blocks + 5
    got = gpu_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), tabs, wl.dec_ctx, wl.scale, 40)
    check_device_error(1)                    # PA_DEVERR_BLOCK_ID
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got[:1], ref[:1], "untouched sequence")


# ------------------------------------------------------- full-size workloads --

def _step(pk, wl, pt=0):
    """reshape_and_cache of this step's tokens, then decode (the hot path)."""
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    if wl.slot_mapping is not None and len(wl.slot_mapping):
        pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    got = gpu_decode(pk, wl.q, kp, vp, wl.dec_tables, wl.dec_ctx, wl.scale,
                     int(wl.dec_ctx.max()), pt)
    return got, kp, vp


def test_mha_7b_full(pk):
    wl = make_workload("mha_7b")
    got, kp, vp = _step(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    assert np.array_equal(host_bits(kp), ek) and np.array_equal(host_bits(vp), ev)
    ref = paged_decode(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale)
    stats = assert_attention_close(got, ref, "mha_7b")
    check_device_error(0)
    print("mha_7b", stats)


def test_gqa_8b_full(pk):
    wl = make_workload("gqa_8b")
    got, kp, vp = _step(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_decode(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale)
    stats = assert_attention_close(got, ref, "gqa_8b")
    check_device_error(0)
    print("gqa_8b", stats)


@pytest.mark.parametrize("pt", [128, 1024])
def test_gqa_8b_other_partition_sizes_sampled(pk, pt):
    wl = make_workload("gqa_8b")
    got, _, _ = _step(pk, wl, pt)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rng = np.random.default_rng(pt)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 24), rng.integers(0, 32, 24))]
    ref = paged_decode_rows(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, rows)
    for (b, h), r in ref.items():
        assert_attention_close(got[b, h], r, f"pt={pt} row {(b, h)}")


def test_gqa_70b_shared_prefix_and_cow(pk):
    """100 sequences share 32 prefix blocks (refcount 100); 10 copy the last
    shared block and write a divergent token into their copy. The other 90
    sequences' outputs must stay bit-identical; the 10 must match the oracle
    on the new state."""
    torch = torch_cuda()
    wl = make_workload("gqa_70b_cow")
    before, kp, vp = _step(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    # every query head of 16 sequences: the 10 that diverge below and 6 others
    rng = np.random.default_rng(3)
    others0 = np.setdiff1d(np.arange(100), wl.cow_seqs)
    seqs = sorted(set(int(b) for b in wl.cow_seqs) | set(int(b) for b in rng.choice(others0, 6, replace=False)))
    assert len(seqs) >= 16
    rows = [(b, h) for b in seqs for h in range(64)]
    ref = paged_decode_rows(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, rows)
    assert_attention_close(np.stack([before[b, h] for b, h in rows]), np.stack([ref[r] for r in rows]),
                           "shared-prefix rows (16 sequences x 64 heads)")
    # copy-on-write of the last shared block for 10 sequences, then a divergent write
    pk.pa_copy_blocks(kp, vp, dev(wl.copy_pairs))
    ek2, ev2 = o_copy(ek, ev, wl.copy_pairs)
    pk.pa_reshape_and_cache(dev(wl.div_k), dev(wl.div_v), kp, vp, dev(wl.div_slots))
    ek2, ev2 = o_rac(wl.div_k, wl.div_v, ek2, ev2, wl.div_slots)
    for blk in list(wl.copy_pairs[:, 1]) + [int(wl.copy_pairs[0, 0])]:
        assert np.array_equal(host_bits(kp[blk]), ek2[blk])
        assert np.array_equal(host_bits(vp[blk]), ev2[blk])
    after = gpu_decode(pk, wl.q, kp, vp, wl.dec_tables_after_cow, wl.dec_ctx, wl.scale, 4096)
    others = np.setdiff1d(np.arange(100), wl.cow_seqs)
    assert np.array_equal(after[others], before[others])
    rows = [(int(b), h) for b in wl.cow_seqs for h in range(64)]
    ref2 = paged_decode_rows(wl.q, ek2, ev2, wl.dec_tables_after_cow, wl.dec_ctx, wl.scale, rows)
    assert_attention_close(np.stack([after[b, h] for b, h in rows]), np.stack([ref2[r] for r in rows]),
                           "diverged rows (10 sequences x 64 heads)")
    for b in wl.cow_seqs:   # the divergent token moves every diverged sequence's outputs
        assert not np.array_equal(after[b], before[b]), f"diverged sequence {int(b)} unchanged"
    check_device_error(0)


def test_mixed_decode_part_full(pk):
    wl = make_workload("mixed")
    got, kp, vp = _step(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_decode(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "mixed decode")
    check_device_error(0)
