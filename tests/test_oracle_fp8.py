"""Pins for the fp8 (E4M3) KV-cache oracle (oracle/fp8.py), on the CPU.

Each pin ties the oracle to something other than itself: torch's own E4M3
type (a library special case), closed forms of the format (exact ties,
subnormals, saturation), the format's error bound, and the bf16 attention
oracle (pinned separately) on values that bf16 represents exactly.
"""
import math

import numpy as np
import pytest

from oracle import attention, fp8
from oracle.bf16 import bf16_bits_to_f64
from workloads import E4M3_NAN, f32_to_bf16_bits, make_decode_case_fp8

torch = pytest.importorskip("torch")


def _torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def test_decode_all_codes_match_torch():
    c = np.arange(256, dtype=np.uint8)
    ours, ref = fp8.e4m3_to_f64(c), _torch_decode(c)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))  # -0 for 0x80
    assert set(np.nonzero(np.isnan(ours))[0]) == {0x7F, 0xFF}


def test_decode_closed_forms():
    v = fp8.e4m3_to_f64(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0xFE, 0xB8], dtype=np.uint8))
    assert list(v) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -448.0, -1.0]


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(11)
    mags = np.exp2(rng.uniform(-12, math.log2(448.0), 200000))
    x = (mags * rng.choice([-1.0, 1.0], mags.shape)).astype(np.float32).astype(np.float64)
    vals = fp8.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2.0                      # every exact tie
    x = np.concatenate([x, mids, -mids, vals, -vals])
    ours = fp8.f64_to_e4m3(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("x,code", [
    (0.0, 0x00), (-0.0, 0x80), (448.0, 0x7E), (-448.0, 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00),          # tie between 0 and the smallest subnormal: even
    (3 * 2.0 ** -10, 0x02),                         # tie between 0x01 and 0x02: even
    (-(2.0 ** -11), 0x80),                          # rounds to zero, sign kept
    (1.0625, 0x38), (1.1875, 0x3A),                 # ties inside a binade: even mantissa
    (0.96875, 0x38),                                # tie across a binade edge: 1.0
    (2.0 ** -6 * 15 / 16, 0x08),                    # between the largest subnormal and 2^-6: tie to even 0x08
    (460.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e30, 0xFE),   # saturate
    (math.inf, 0x7E), (-math.inf, 0xFE), (math.nan, 0x7F),
])
def test_encode_closed_forms(x, code):
    assert int(fp8.f64_to_e4m3(np.array([x]))[0]) == code


def test_encode_decode_round_trip():
    c = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.f64_to_e4m3(fp8.e4m3_to_f64(c)), c)


def test_quantize_divides_in_fp32_by_the_scale():
    # power-of-two scales: the quotient is exact, so quantize == encode(x * 2^-k)
    rng = np.random.default_rng(3)
    bits = f32_to_bf16_bits(rng.standard_normal((64, 128), dtype=np.float32))
    x = bf16_bits_to_f64(bits)
    for k in (-7, -5, 0, 3):
        assert np.array_equal(fp8.quantize(bits, np.float32(2.0 ** k)), fp8.f64_to_e4m3(x * 2.0 ** -k))
    # x = 1, scale = 3.368421 (fp32): the fp32 quotient is exactly 0.296875,
    # the midpoint of 0x29 (0.28125) and 0x2A (0.3125), so the code is the
    # even 0x2A; the exact quotient lies just below the midpoint (an fp64
    # division would give 0x29)
    s = np.float32(3.368421)
    assert float(np.float32(1.0) / s) == 0.296875 and 1.0 / float(s) < 0.296875
    assert int(fp8.quantize(f32_to_bf16_bits(np.array([1.0], np.float32)), s)[0]) == 0x2A


def test_quantization_error_within_format_bound():
    """|dequant(quant(x)) - x| <= half an ulp of E4M3 at x/scale, times scale:
    2^-4 relative in the normal range, 2^-10 absolute below 2^-6."""
    rng = np.random.default_rng(5)
    bits = f32_to_bf16_bits(rng.standard_normal((4096,), dtype=np.float32) * 3)
    x = bf16_bits_to_f64(bits)
    s = np.float32(2.0 ** -6 * 1.37)
    y = fp8.dequantize(fp8.quantize(bits, s), float(s))
    q = x / float(s)
    inr = np.abs(q) <= 448.0
    assert inr.sum() > 4000 and (~inr).sum() > 0       # both regimes are exercised
    bound = np.where(np.abs(q) >= 2.0 ** -6, np.abs(q) * 2.0 ** -4, 2.0 ** -10) * float(s) * (1 + 1e-6)
    assert np.all(np.abs(y - x)[inr] <= bound[inr])
    # beyond the largest magnitude the code saturates: y = sign(x) * 448 * scale
    assert np.array_equal(y[~inr], np.sign(x[~inr]) * 448.0 * float(s))


def test_cache_write_round_trip_and_skips():
    wl = make_decode_case_fp8(21, [5, 16, 17, 40], 8, 2, 64, n_new=1)
    slots = wl.slot_mapping.copy()
    slots[1] = -1                                             # padding row
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    kp, vp = fp8.reshape_and_cache_fp8(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, slots, ks, vs)
    changed = np.nonzero(np.any(kp != wl.k_pool, axis=(1, 3)) | np.any(vp != wl.v_pool, axis=(1, 3)))
    for t, s in enumerate(slots):
        blk, off = divmod(int(s), 16)
        if s < 0:
            continue
        for h in range(wl.n_kv_heads):
            assert np.array_equal(kp[blk, h, off], fp8.quantize(wl.new_k[t, h], ks[h]))
            assert np.array_equal(vp[blk, h, off], fp8.quantize(wl.new_v[t, h], vs[h]))
    # nothing else moved: the slot of the skipped row still holds the fill
    blk, off = divmod(int(wl.slot_mapping[1]), 16)
    assert np.all(kp[blk, :, off] == E4M3_NAN)
    assert len(changed[0]) <= 3 * wl.n_kv_heads


def test_fp8_decode_equals_bf16_oracle_on_exact_values():
    """With power-of-two scales every dequantised value is a bf16 number, so
    the fp8 path must equal the (separately pinned) bf16 paged decode on a
    bf16 pool holding those values, exactly."""
    wl = make_decode_case_fp8(22, [1, 15, 16, 37, 200], 8, 2, 64, n_new=0)
    ks = np.array([2.0 ** -5, 2.0 ** -7], np.float32)
    vs = np.array([2.0 ** -6, 2.0 ** -4], np.float32)
    ref_pool_k = np.empty(wl.k_pool.shape, np.uint16)
    ref_pool_v = np.empty(wl.v_pool.shape, np.uint16)
    for h in range(2):
        dk = fp8.dequantize(wl.k_pool[:, h], float(ks[h])).astype(np.float32)
        dv = fp8.dequantize(wl.v_pool[:, h], float(vs[h])).astype(np.float32)
        ref_pool_k[:, h] = np.where(np.isnan(dk), 0x7FC0, f32_to_bf16_bits(np.nan_to_num(dk)))
        ref_pool_v[:, h] = np.where(np.isnan(dv), 0x7FC0, f32_to_bf16_bits(np.nan_to_num(dv)))
    got = fp8.paged_decode_fp8(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, ks, vs)
    ref = attention.paged_decode(wl.q, ref_pool_k, ref_pool_v, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert np.array_equal(got, ref)


def test_fp8_decode_matches_torch_sdpa_with_torch_dequant():
    wl = make_decode_case_fp8(23, [3, 33, 129], 8, 2, 128, n_new=0)
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    got = fp8.paged_decode_fp8(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, ks, vs)
    F = torch.nn.functional
    for b, n in enumerate(wl.dec_ctx):
        n = int(n)
        kc = attention.gather_kv(wl.k_pool, wl.dec_tables[b], n)     # codes [n][Hk][D]
        vc = attention.gather_kv(wl.v_pool, wl.dec_tables[b], n)
        k = _torch_decode(kc) * ks[None, :, None].astype(np.float64)
        v = _torch_decode(vc) * vs[None, :, None].astype(np.float64)
        qb = torch.from_numpy(bf16_bits_to_f64(wl.q[b]))[None, :, None, :]      # [1][H][1][D]
        kt = torch.from_numpy(k.transpose(1, 0, 2).copy())[None]                   # [1][Hk][n][D]
        vt = torch.from_numpy(v.transpose(1, 0, 2).copy())[None]
        ref = F.scaled_dot_product_attention(qb, kt, vt, scale=wl.scale, enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-11, atol=1e-12)


def test_fp8_rows_equal_full():
    wl = make_decode_case_fp8(24, [40, 70], 8, 2, 64, n_new=0)
    ks, vs = wl.meta["k_scale"], wl.meta["v_scale"]
    full = fp8.paged_decode_fp8(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, ks, vs)
    rows = [(0, 0), (1, 7), (1, 3)]
    part = fp8.paged_decode_fp8_rows(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale,
                                     ks, vs, rows)
    for r in rows:
        assert np.array_equal(part[r], full[r])
