"""GPU parity for sliding-window decode against the fp64 oracle.

Tolerance per element: |gpu - ref| <= 2e-3 + 1e-2 * |ref|. Tables hold -1 for
the blocks wholly before each window (released), so a kernel that read one
would fault its bounds check (flag) or read NaN; windows from 0 (the newest
token only) through block edges to wider than the context.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode_window
from oracle.cache_ops import reshape_and_cache as o_rac
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_decode_case_window, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def run(pk, wl, window, pt=0, decode_fn="window"):
    torch = torch_cuda()
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    q = dev(wl.q)
    out = torch.full_like(q, 0x7FC0)
    n, H, D = q.shape
    max_ctx = int(wl.dec_ctx.max())
    wsb = pk.pa_decode_workspace_bytes(n, H, D, max_ctx, pt)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
    if decode_fn == "window":
        pk.pa_decode_window(out, q, kp, vp, dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale, max_ctx, window,
                            workspace=ws, partition_tokens=pt)
    else:
        pk.pa_decode(out, q, kp, vp, dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale, max_ctx,
                     workspace=ws, partition_tokens=pt)
    torch.cuda.synchronize()
    return host_bits(out)


def oracle(wl, window):
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    return paged_decode_window(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, window)


@pytest.mark.parametrize("window", [0, 1, 15, 16, 17, 100, 600])
@pytest.mark.parametrize("D,H,Hk", [(128, 32, 8), (64, 8, 8), (128, 16, 2)])
@pytest.mark.parametrize("pt", [0, 64])
def test_window_decode(pk, window, D, H, Hk, pt):
    ctx = [1, 2, 16, 17, 40, 129, 300, 513, 1000]
    wl = make_decode_case_window(600 + window + D + H + pt, ctx, H, Hk, D, window)
    got = run(pk, wl, window, pt)
    assert_attention_close(got, oracle(wl, window), f"window={window} D={D} H={H} Hk={Hk} pt={pt}")
    check_device_error(0)


def test_wide_window_equals_full_decode_bit_for_bit(pk):
    wl = make_decode_case(650, [1, 15, 16, 300, 1000], 32, 8, 128, n_new=1)
    a = run(pk, wl, 5000)
    b = run(pk, wl, 0, decode_fn="full")
    assert np.array_equal(a, b)
    check_device_error(0)


def test_swa_mistral_sampled_rows(pk):
    wl = make_workload("swa_mistral")
    W = wl.meta["window"]
    got = run(pk, wl, W)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rng = np.random.default_rng(11)
    seqs = [int(b) for b in rng.integers(0, len(wl.dec_ctx), 6)] + [int(np.argmax(wl.dec_ctx))]
    for b in seqs:
        sub = slice(b, b + 1)
        ref = paged_decode_window(wl.q[sub], ek, ev, wl.dec_tables[sub], wl.dec_ctx[sub], wl.scale, W)
        for h in (0, 7, 31):
            assert_attention_close(got[b, h], ref[0, h], f"swa row {(b, h)}")
    check_device_error(0)
