"""GPU parity for the tensor-core decode kernel (pa_decode_tc: warp-level MMAs
for QK^T and PV, TMA-staged swizzled tiles) against the fp64 oracle, at every
group size; pa_decode takes this kernel by itself for groups of 8 at
head_dim 128.

Tolerance (per element): |gpu - ref| <= 2e-3 + 1e-2 * |ref|. Cases: groups
1, 2, 4, 8; contexts 1, 15, 16, 17 and ragged tails with NaN-poisoned slots
past the context; partitions of 64, 512 and 2048 tokens (one to many per
row); logits of order +-100; zero contexts; permuted physical blocks (bit
identical); a bad block id; sampled rows of the 8B batch.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode, paged_decode_rows
from oracle.cache_ops import reshape_and_cache as o_rac
from tests._gpu import assert_attention_close, bf16_to_f64, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def tc_decode(pk, q, kp, vp, tables, ctx, scale, max_ctx, pt=0):
    torch = torch_cuda()
    q_d = q if not isinstance(q, np.ndarray) else dev(q)
    out = torch.empty_like(q_d)
    n_seqs, H, D = q_d.shape
    ws_bytes = pk.pa_decode_workspace_bytes(n_seqs, H, D, max_ctx, pt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    pk.pa_decode_tc(out, q_d, kp, vp, tables if not isinstance(tables, np.ndarray) else dev(tables),
                    ctx if not isinstance(ctx, np.ndarray) else dev(ctx), scale, max_ctx,
                    workspace=ws, partition_tokens=pt)
    torch.cuda.synchronize()
    return host_bits(out)


@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 4), (16, 4), (64, 8)])
@pytest.mark.parametrize("pt", [0, 64, 2048])
def test_groups_and_partitions(pk, H, Hk, pt):
    ctx = [1, 15, 16, 17, 37, 64, 129, 300, 513, 1000, 2500]
    wl = make_decode_case(900 + H + Hk + pt, ctx, H, Hk, 128)
    got = tc_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx, wl.scale, max(ctx), pt)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, f"tc H={H} Hk={Hk} pt={pt}")
    check_device_error(0)


def test_context_one_is_exact(pk):
    """One visible token: out = v0 exactly (p = 1 in both terms, O / l = v0)."""
    wl = make_decode_case(920, [1, 1, 1], 32, 8, 128)
    got = tc_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx, wl.scale, 1)
    for b in range(3):
        v0 = wl.v_pool[wl.dec_tables[b, 0], :, 0, :]          # [Hk][D]
        assert np.array_equal(got[b], np.repeat(v0, 4, axis=0))


@pytest.mark.parametrize("H,Hk", [(32, 8), (64, 8)])
def test_hot_logits_and_zero_contexts(pk, H, Hk):
    wl = make_decode_case(921, [0, 77, 500, 1, 0], H, Hk, 128)
    qf = bf16_to_f64(wl.q) * 20.0
    q_hot = ((qf.astype(np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    got = tc_decode(pk, q_hot, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx, wl.scale, 500, 128)
    assert np.all(got[0] == 0) and np.all(got[4] == 0)
    ref = paged_decode(q_hot, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "tc hot")
    check_device_error(0)


def test_block_permutation_gives_identical_bits(pk):
    wl = make_decode_case(922, [40, 300, 1000, 16], 64, 8, 128)
    a = tc_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), wl.dec_tables, wl.dec_ctx, wl.scale, 1000, 256)
    pi = np.random.default_rng(11).permutation(wl.num_blocks)
    kp = np.empty_like(wl.k_pool)
    vp = np.empty_like(wl.v_pool)
    kp[pi] = wl.k_pool
    vp[pi] = wl.v_pool
    tabs = np.where(wl.dec_tables >= 0, pi[np.maximum(wl.dec_tables, 0)], -1).astype(np.int32)
    b = tc_decode(pk, wl.q, dev(kp), dev(vp), tabs, wl.dec_ctx, wl.scale, 1000, 256)
    assert np.array_equal(a, b)


def test_bad_block_id_is_flagged_not_faulted(pk):
    wl = make_decode_case(923, [40, 40], 32, 8, 128)
    tabs = wl.dec_tables.copy()
    tabs[1, 1] = wl.num_blocks + 5
    got = tc_decode(pk, wl.q, dev(wl.k_pool), dev(wl.v_pool), tabs, wl.dec_ctx, wl.scale, 40)
    check_device_error(1)                    # PA_DEVERR_BLOCK_ID
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got[:1], ref[:1], "untouched sequence")


def test_gqa_8b_sampled_rows(pk):
    wl = make_workload("gqa_8b")
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    got = tc_decode(pk, wl.q, kp, vp, wl.dec_tables, wl.dec_ctx, wl.scale, int(wl.dec_ctx.max()))
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rng = np.random.default_rng(12)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 24), rng.integers(0, 32, 24))]
    ref = paged_decode_rows(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, rows)
    for (b, h), r in ref.items():
        assert_attention_close(got[b, h], r, f"tc 8B row {(b, h)}")
    check_device_error(0)
