"""GPU parity for the fp8 (E4M3) KV cache: the cache write against the oracle
bit for bit, and decode over an fp8 cache against the fp64 oracle.

Decode tolerance is the bf16 path's, per element: |gpu - ref| <= 2e-3 +
1e-2 * |ref| (the oracle attends over the exact dequantised values, so the
fp8 rounding itself is part of the input, not of the error). Cached codes
are drawn uniformly over all finite E4M3 patterns (zeros, subnormals, up to
+-448), unused slots hold E4M3 NaN, so a read of an unwritten slot shows.
"""
import numpy as np
import pytest

from oracle.fp8 import (e4m3_to_f64, paged_decode_fp8, paged_decode_fp8_rows, quantize,
                        reshape_and_cache_fp8)
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import E4M3_NAN, f32_to_bf16_bits, make_decode_case_fp8, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def _scales(wl):
    return dev(wl.meta["k_scale"]), dev(wl.meta["v_scale"])


def gpu_write(pk, wl, new_k=None, new_v=None, slots=None):
    torch = torch_cuda()
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    ks, vs = _scales(wl)
    pk.pa_reshape_and_cache_fp8(dev(wl.new_k if new_k is None else new_k),
                                dev(wl.new_v if new_v is None else new_v), kp, vp,
                                dev(wl.slot_mapping if slots is None else slots), ks, vs)
    torch.cuda.synchronize()
    return kp, vp


def gpu_decode(pk, wl, kp, vp, pt=0):
    torch = torch_cuda()
    q = dev(wl.q)
    out = torch.full_like(q, 0x7FC0)
    n, H, D = q.shape
    max_ctx = int(wl.dec_ctx.max())
    wsb = pk.pa_decode_workspace_bytes(n, H, D, max_ctx, pt)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
    ks, vs = _scales(wl)
    pk.pa_decode_fp8(out, q, kp, vp, ks, vs, dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale, max_ctx,
                     workspace=ws, partition_tokens=pt)
    torch.cuda.synchronize()
    return host_bits(out)


@pytest.mark.parametrize("D,Hk", [(64, 2), (128, 8)])
def test_cache_write_bit_exact(pk, D, Hk):
    wl = make_decode_case_fp8(300 + D, [1, 15, 16, 17, 37, 100], 2 * Hk, Hk, D, n_new=1)
    kp, vp = gpu_write(pk, wl)
    ek, ev = reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping,
                                   wl.meta["k_scale"], wl.meta["v_scale"])
    assert np.array_equal(kp.cpu().numpy(), ek)
    assert np.array_equal(vp.cpu().numpy(), ev)
    check_device_error(0)


def test_cache_write_saturation_ties_subnormals_skips(pk):
    """New values chosen to hit every corner of the encoding: exact ties of
    the fp32 quotient, values that round to zero (both signs), subnormals,
    and magnitudes beyond 448 * scale (saturate); one padding row."""
    wl = make_decode_case_fp8(310, [20, 40, 60, 80], 8, 2, 128, n_new=1)
    ks = np.array([2.0 ** -3, 2.0 ** -6], np.float32)          # exact quotients
    wl.meta["k_scale"], wl.meta["v_scale"] = ks, ks
    vals = e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2.0                        # ties of the quotient
    pool = np.concatenate([mids, -mids, vals, [1e3, -1e3, 5e4, -5e4, 2.0 ** -12, -(2.0 ** -12)]])
    rng = np.random.default_rng(0)
    for arr in (wl.new_k, wl.new_v):
        for t in range(arr.shape[0]):
            for h in range(2):
                x = rng.choice(pool, size=128) * float(ks[h])
                arr[t, h] = f32_to_bf16_bits(x.astype(np.float32))
    slots = wl.slot_mapping.copy()
    slots[2] = -1
    kp, vp = gpu_write(pk, wl, slots=slots)
    ek, ev = reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, slots, ks, ks)
    assert np.array_equal(kp.cpu().numpy(), ek)
    assert np.array_equal(vp.cpu().numpy(), ev)
    codes = ek[np.asarray(wl.slot_mapping[[0, 1, 3]]) // 16]
    assert (codes == 0x7E).any() and (codes == 0xFE).any()       # saturation was exercised
    blk, off = divmod(int(wl.slot_mapping[2]), 16)
    assert np.all(kp.cpu().numpy()[blk, :, off] == E4M3_NAN)   # the padding row wrote nothing
    check_device_error(0)


def test_cache_write_bad_slot_sets_flag(pk):
    wl = make_decode_case_fp8(311, [20, 40], 8, 2, 128, n_new=1)
    slots = wl.slot_mapping.copy()
    slots[1] = wl.num_blocks * 16 + 5
    kp, _ = gpu_write(pk, wl, slots=slots)
    check_device_error(2)  # PA_DEVERR_SLOT
    ek, _ = reshape_and_cache_fp8(wl.new_k[:1], wl.new_v[:1], wl.k_pool, wl.v_pool, slots[:1],
                                  wl.meta["k_scale"], wl.meta["v_scale"])
    assert np.array_equal(kp.cpu().numpy(), ek)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("pt", [0, 64])
def test_decode_shapes_groups_partitions(pk, D, H, Hk, pt):
    ctx = [1, 15, 16, 17, 37, 129, 300, 513, 1000]
    wl = make_decode_case_fp8(400 + D + H + Hk + pt, ctx, H, Hk, D, n_new=1)
    kp, vp = gpu_write(pk, wl)
    got = gpu_decode(pk, wl, kp, vp, pt)
    ek, ev = reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping,
                                   wl.meta["k_scale"], wl.meta["v_scale"])
    ref = paged_decode_fp8(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, wl.meta["k_scale"],
                           wl.meta["v_scale"])
    assert_attention_close(got, ref, f"fp8 D={D} H={H} Hk={Hk} pt={pt}")
    check_device_error(0)


def test_decode_context_one_is_v0(pk):
    """One cached token: the output is its V row exactly (weight 1), i.e. the
    bf16 rounding of decode(code) * v_scale."""
    wl = make_decode_case_fp8(420, [1, 1], 8, 2, 128, n_new=1)
    kp, vp = gpu_write(pk, wl)
    got = gpu_decode(pk, wl, kp, vp)
    ek, ev = reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping,
                                   wl.meta["k_scale"], wl.meta["v_scale"])
    for b in range(2):
        blk, off = divmod(int(wl.slot_mapping[b]), 16)
        for h in range(8):
            v0 = e4m3_to_f64(ev[blk, h // 4, off]) * float(wl.meta["v_scale"][h // 4])
            assert np.array_equal(got[b, h], f32_to_bf16_bits(v0.astype(np.float32)))


def test_gqa_8b_fp8_sampled_rows(pk):
    wl = make_workload("gqa_8b_fp8")
    kp, vp = gpu_write(pk, wl)
    got = gpu_decode(pk, wl, kp, vp)
    # the oracle's view of the pools after the write: only the 64 written slots changed
    ek, ev = reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping,
                                   wl.meta["k_scale"], wl.meta["v_scale"])
    assert np.array_equal(kp.cpu().numpy(), ek)
    rng = np.random.default_rng(7)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 40), rng.integers(0, 32, 40))]
    rows += [(int(np.argmax(wl.dec_ctx)), 31), (int(np.argmin(wl.dec_ctx)), 0)]
    ref = paged_decode_fp8_rows(wl.q, ek, ev, wl.dec_tables, wl.dec_ctx, wl.scale, wl.meta["k_scale"],
                                wl.meta["v_scale"], rows)
    for r in rows:
        assert_attention_close(got[r], ref[r], f"gqa_8b_fp8 row {r}")
    check_device_error(0)


def test_fp8_quantisation_error_against_bf16_reference(pk):
    """Property at full scale: the fp8 cache write of bf16 K/V, decoded, stays
    within the format's half-ulp bound of the bf16 inputs (2^-4 relative)."""
    wl = make_decode_case_fp8(430, [64] * 8, 32, 8, 128, n_new=1)
    kp, _ = gpu_write(pk, wl)
    codes = kp.cpu().numpy()
    for t, s in enumerate(wl.slot_mapping):
        blk, off = divmod(int(s), 16)
        for h in range(8):
            x = (wl.new_k[t, h].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            y = e4m3_to_f64(codes[blk, h, off]) * float(wl.meta["k_scale"][h])
            q = np.abs(x) / float(wl.meta["k_scale"][h])
            bound = np.where(q >= 2.0 ** -6, q * 2.0 ** -4, 2.0 ** -10) * float(wl.meta["k_scale"][h])
            assert np.all(np.abs(y - x) <= bound * (1 + 1e-6))
            assert np.array_equal(codes[blk, h, off], quantize(wl.new_k[t, h], wl.meta["k_scale"][h]))
