"""pa_decode_planned: decode from a host-built plan (pa_decode_plan).

A plan only reorders which CTA computes which (partition, KV head,
sequence), so the outputs must be bit-identical to the unplanned call's on
every kernel: the CUDA-core kernel (groups up to 4, head_dim 64 and 128, with
a window), the tensor-core kernel (group 8) and the E4M3 cache. Contexts
include 0 (a zero row), 1 and lengths around partition edges. A plan item
outside the call's bounds is flagged and skipped.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_decode_case_fp8

pytestmark = pytest.mark.gpu

PA_DEVERR_PLAN = 128


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


CTX = [1, 0, 17, 300, 511, 512, 513, 1000, 2049, 4000, 64, 1025]


def _plan(pk, wl, max_ctx, window=-1, eb=2, pt=0):
    items = pk.pa_decode_plan(wl.dec_ctx, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.dec_tables.shape[1],
                              max_ctx, wl.num_blocks, window=window, elem_bytes=eb, partition_tokens=pt)
    return dev(np.ascontiguousarray(items))


@pytest.mark.parametrize("H,Hk,D,pt,window", [(32, 8, 128, 0, -1), (32, 8, 128, 64, -1), (64, 8, 128, 0, -1),
                                               (16, 16, 64, 0, -1), (32, 8, 128, 0, 700)])
def test_planned_equals_unplanned(pk, H, Hk, D, pt, window):
    torch = torch_cuda()
    wl = make_decode_case(900 + H + D + pt + max(window, 0), CTX, H, Hk, D)
    max_ctx = max(CTX)
    q, kp, vp, tabs, ctx = dev(wl.q), dev(wl.k_pool), dev(wl.v_pool), dev(wl.dec_tables), dev(wl.dec_ctx)
    ws = pk.decode_workspace(q, max_ctx, pt)
    out_a = torch.full_like(q, 0x7FC0)
    out_b = torch.full_like(q, 0x7FC0)
    if window >= 0:
        pk.pa_decode_window(out_a, q, kp, vp, tabs, ctx, wl.scale, max_ctx, window, workspace=ws, partition_tokens=pt)
    else:
        pk.pa_decode(out_a, q, kp, vp, tabs, ctx, wl.scale, max_ctx, workspace=ws, partition_tokens=pt)
    items = _plan(pk, wl, max_ctx, window=window, pt=pt)
    pk.pa_decode_planned(out_b, q, kp, vp, tabs, ctx, wl.scale, max_ctx, items, window=window, workspace=ws,
                         partition_tokens=pt)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out_a), host_bits(out_b)), "a plan changed the results"
    if window < 0:
        ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
        assert_attention_close(host_bits(out_b), ref, f"planned decode H={H} Hk={Hk} D={D} pt={pt}")
    check_device_error(0)


def test_planned_fp8_equals_unplanned(pk):
    torch = torch_cuda()
    wl = make_decode_case_fp8(950, CTX, 32, 8, 128, n_new=0)
    max_ctx = max(CTX)
    q, kp, vp, tabs, ctx = dev(wl.q), dev(wl.k_pool), dev(wl.v_pool), dev(wl.dec_tables), dev(wl.dec_ctx)
    ks, vs = dev(wl.meta["k_scale"]), dev(wl.meta["v_scale"])
    ws = pk.decode_workspace(q, max_ctx)
    out_a = torch.full_like(q, 0x7FC0)
    out_b = torch.full_like(q, 0x7FC0)
    pk.pa_decode_fp8(out_a, q, kp, vp, ks, vs, tabs, ctx, wl.scale, max_ctx, workspace=ws)
    items = _plan(pk, wl, max_ctx, eb=1)
    pk.pa_decode_planned(out_b, q, kp, vp, tabs, ctx, wl.scale, max_ctx, items, k_scale=ks, v_scale=vs,
                         workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out_a), host_bits(out_b)), "a plan changed the E4M3 results"
    check_device_error(0)


def test_plan_item_out_of_bounds_is_flagged(pk):
    torch = torch_cuda()
    wl = make_decode_case(960, CTX, 32, 8, 128)
    max_ctx = max(CTX)
    q, kp, vp, tabs, ctx = dev(wl.q), dev(wl.k_pool), dev(wl.v_pool), dev(wl.dec_tables), dev(wl.dec_ctx)
    ws = pk.decode_workspace(q, max_ctx)
    items = pk.pa_decode_plan(wl.dec_ctx, 32, 8, 128, wl.dec_tables.shape[1], max_ctx, wl.num_blocks)
    bad = np.array([[0, 0, len(CTX), 0], [0, 8, 0, 0], [-1, 0, 0, 0]], dtype=np.int32)  # sequence, kv head, partition
    out = torch.full_like(q, 0x7FC0)
    pk.pa_decode_planned(out, q, kp, vp, tabs, ctx, wl.scale, max_ctx, dev(np.concatenate([items, bad])),
                         workspace=ws)
    torch.cuda.synchronize()
    check_device_error(PA_DEVERR_PLAN)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(host_bits(out), ref, "valid items of a plan with bad ones")
