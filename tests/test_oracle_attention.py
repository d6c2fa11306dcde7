"""Pins for the fp64 attention oracle (CPU only).

Each test ties the oracle to something other than itself: torch's
scaled_dot_product_attention on contiguous tensors drawn independently of the
paged layout, closed-form special cases, invariances the pages state, and a
pure-Python brute force on the tiny workload.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle.bf16 import bf16_bits_to_f64
from workloads import make_decode_case, make_prefill_case, make_workload


def _sdpa_decode(wl):
    """torch SDPA in fp64 over each sequence's contiguous K/V (from the
    generator's logical arrays, never through the paged pool)."""
    outs = []
    for b in range(len(wl.dec_ctx)):
        q = torch.from_numpy(bf16_bits_to_f64(wl.q[b]))[None, :, None, :]          # [1,H,1,D]
        k = torch.from_numpy(bf16_bits_to_f64(wl.seq_k[b])).permute(1, 0, 2)[None]  # [1,Hk,T,D]
        v = torch.from_numpy(bf16_bits_to_f64(wl.seq_v[b])).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, scale=wl.scale, enable_gqa=(wl.n_heads != wl.n_kv_heads))
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


def _pools_with_new_tokens(wl):
    """Pools after this step's tokens are written (plain numpy scatter)."""
    from oracle.cache_ops import reshape_and_cache
    return reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)


@pytest.mark.parametrize("case", [
    dict(ctx=[1, 15, 16, 37], H=4, Hk=4, D=64),
    dict(ctx=[17, 3, 64, 100, 33], H=8, Hk=2, D=64),
    dict(ctx=[40, 1, 129], H=8, Hk=1, D=128),
    dict(ctx=[50, 16], H=16, Hk=2, D=128),
])
def test_decode_equals_sdpa_on_contiguous(case):
    wl = make_decode_case(11, case["ctx"], case["H"], case["Hk"], case["D"], n_new=1)
    kp, vp = _pools_with_new_tokens(wl)
    got = A.paged_decode(wl.q, kp, vp, wl.dec_tables, wl.dec_ctx, wl.scale)
    ref = _sdpa_decode(wl)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_tiny_workload_equals_sdpa():
    wl = make_workload("tiny_mha", keep_logical=True)
    got = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    np.testing.assert_allclose(got, _sdpa_decode(wl), rtol=1e-12, atol=1e-13)
    assert np.isfinite(got).all()          # never touched a NaN-poisoned slot


def test_tiny_workload_brute_force_python():
    """Pure-Python loops with math.fsum and math.exp; no numpy arithmetic."""
    wl = make_workload("tiny_mha", keep_logical=True)
    got = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)

    def f(bits):
        return float(bf16_bits_to_f64(np.array([bits], dtype=np.uint16))[0])

    for b, n in enumerate(wl.dec_ctx):
        K = wl.seq_k[b]
        V = wl.seq_v[b]
        for h in range(wl.n_heads):
            qv = [f(x) for x in wl.q[b, h]]
            s = [wl.scale * math.fsum(qv[d] * f(K[t, h, d]) for d in range(wl.head_dim))
                 for t in range(n)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for d in range(wl.head_dim):
                ref = math.fsum(e[t] * f(V[t, h, d]) for t in range(n)) / z
                assert abs(got[b, h, d] - ref) <= 1e-12 * (1 + abs(ref))


def test_context_one_returns_v0_exactly():
    wl = make_decode_case(5, [1, 1, 1], 8, 2, 128)
    got = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    for b in range(3):
        for h in range(8):
            v0 = bf16_bits_to_f64(wl.seq_v[b][0, h // 4])
            assert np.array_equal(got[b, h], v0)


def test_equal_keys_and_zero_scale_give_mean_of_v():
    wl = make_decode_case(6, [23, 48], 4, 4, 64)
    # scale 0: every score is 0, weights uniform
    got = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, 0.0)
    for b in range(2):
        mean = bf16_bits_to_f64(wl.seq_v[b]).mean(axis=0)     # [Hk][D]
        np.testing.assert_allclose(got[b], mean, rtol=1e-13, atol=1e-15)
    # all keys equal: same scores, uniform weights, whatever q is
    kp = wl.k_pool.copy()
    for b in range(2):
        for blk in wl.dec_tables[b][wl.dec_tables[b] >= 0]:
            kp[blk] = wl.seq_k[b][0][:, None, :]
    got = A.paged_decode(wl.q, kp, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    for b in range(2):
        mean = bf16_bits_to_f64(wl.seq_v[b]).mean(axis=0)
        np.testing.assert_allclose(got[b], mean, rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    """q aligned with one key at a huge scale: softmax is one-hot on it."""
    wl = make_decode_case(7, [37], 2, 2, 64)
    kp = wl.k_pool.copy()
    t_hot = 21
    blk, off = wl.dec_tables[0][t_hot // 16], t_hot % 16
    kp[blk, :, off, :] = wl.q[0]                 # k_hot = q, so q.k_hot = |q|^2
    got = A.paged_decode(wl.q, kp, wl.v_pool, wl.dec_tables, wl.dec_ctx, 50.0)
    for h in range(2):
        np.testing.assert_allclose(got[0, h], bf16_bits_to_f64(wl.seq_v[0][t_hot, h]), atol=1e-12)


def test_invariant_under_physical_block_permutation():
    """Blocks 'can be physically non-contiguous': relabelling physical ids
    (pool and tables together) cannot change the result."""
    wl = make_decode_case(8, [5, 16, 17, 80, 33], 8, 2, 64)
    ref = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    rng = np.random.default_rng(123)
    pi = rng.permutation(wl.num_blocks)
    kp = np.empty_like(wl.k_pool)
    vp = np.empty_like(wl.v_pool)
    kp[pi] = wl.k_pool
    vp[pi] = wl.v_pool
    tabs = np.where(wl.dec_tables >= 0, pi[np.maximum(wl.dec_tables, 0)], -1)
    got = A.paged_decode(wl.q, kp, vp, tabs, wl.dec_ctx, wl.scale)
    assert np.array_equal(got, ref)


def test_paged_equals_unpaged_contiguous_layout():
    """The same tokens laid out contiguously (table = 0,1,2,...) give the same output."""
    wl = make_decode_case(9, [31, 64, 7], 8, 4, 128)
    ref = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    for b in range(3):
        n = int(wl.dec_ctx[b])
        nb = (n + 15) // 16
        kp = np.zeros((nb, wl.n_kv_heads, 16, wl.head_dim), np.uint16)
        vp = np.zeros_like(kp)
        for t in range(n):
            kp[t // 16, :, t % 16] = wl.seq_k[b][t]
            vp[t // 16, :, t % 16] = wl.seq_v[b][t]
        got = A.paged_decode(wl.q[b:b + 1], kp, vp, np.arange(nb, dtype=np.int32)[None],
                             wl.dec_ctx[b:b + 1], wl.scale)
        assert np.array_equal(got[0], ref[b])


def test_zero_context_gives_zero_row():
    wl = make_decode_case(10, [3, 5], 4, 2, 64)
    ctx = wl.dec_ctx.copy()
    ctx[1] = 0
    got = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, ctx, wl.scale)
    assert np.all(got[1] == 0.0)


def test_score_shift_invariance():
    """Adding the same offset vector c to every key adds q.c to every score of
    a head, which the softmax cancels."""
    wl = make_decode_case(12, [29], 2, 1, 64)
    base = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    kf = bf16_bits_to_f64(wl.k_pool)
    kf = np.where(np.isnan(kf), 0.0, kf) + 0.25       # c = 0.25 * ones
    got = A.paged_decode(wl.q, kf, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    np.testing.assert_allclose(got, base, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- prefill --

def _sdpa_causal_full(k_seq, v_seq, q_rows, scale, g):
    """Causal SDPA over a whole sequence (square mask, torch's is_causal)."""
    q = torch.from_numpy(q_rows).permute(1, 0, 2)[None]          # [1,H,T,D]
    k = torch.from_numpy(k_seq).permute(1, 0, 2)[None]
    v = torch.from_numpy(v_seq).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale,
                                                         enable_gqa=(g > 1))
    return o[0].permute(1, 0, 2).numpy()                           # [T,H,D]


@pytest.mark.parametrize("case", [
    dict(pctx=[40], plen=[40], H=4, Hk=4, D=64),        # whole prompt as one chunk
    dict(pctx=[70, 33], plen=[20, 33], H=8, Hk=2, D=64),  # chunk at an offset
    dict(pctx=[129], plen=[17], H=4, Hk=1, D=128),
])
def test_prefill_chunk_equals_rows_of_full_causal_sdpa(case):
    wl = make_prefill_case(21, case["pctx"], case["plen"], [], case["H"], case["Hk"], case["D"])
    from oracle.cache_ops import reshape_and_cache
    kp, vp = reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    got = A.paged_prefill(wl.q_pf, kp, vp, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    g = case["H"] // case["Hk"]
    rng = np.random.default_rng(5)
    for s in range(len(case["pctx"])):
        n, L = case["pctx"][s], case["plen"][s]
        r0 = int(wl.q_start_loc[s])
        # full-length query block: random rows for the earlier positions, the
        # chunk's own queries for the last L positions
        qfull = rng.standard_normal((n, case["H"], case["D"]))
        qfull[n - L:] = bf16_bits_to_f64(wl.q_pf[r0:r0 + L])
        ref = _sdpa_causal_full(bf16_bits_to_f64(wl.seq_k[s]), bf16_bits_to_f64(wl.seq_v[s]),
                                qfull, wl.scale, g)
        np.testing.assert_allclose(got[r0:r0 + L], ref[n - L:], rtol=1e-12, atol=1e-13)


def test_prefill_last_row_equals_decode():
    wl = make_prefill_case(22, [52], [9], [], 8, 2, 64)
    from oracle.cache_ops import reshape_and_cache
    kp, vp = reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    pf = A.paged_prefill(wl.q_pf, kp, vp, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    dec = A.paged_decode(wl.q_pf[8:9], kp, vp, wl.pf_tables, wl.pf_ctx, wl.scale)
    assert np.array_equal(pf[8], dec[0])
    # the first chunk row sees exactly ctx - L + 1 tokens
    dec0 = A.paged_decode(wl.q_pf[0:1], kp, vp, wl.pf_tables, np.array([52 - 9 + 1]), wl.scale)
    assert np.array_equal(pf[0], dec0[0])


def test_prefill_sampled_rows_match_full():
    wl = make_prefill_case(23, [45, 20], [13, 20], [], 4, 2, 64)
    from oracle.cache_ops import reshape_and_cache
    kp, vp = reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    full = A.paged_prefill(wl.q_pf, kp, vp, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    rows = [(0, 1), (12, 3), (13, 0), (32, 2)]
    part = A.paged_prefill(wl.q_pf, kp, vp, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale,
                           rows=rows)
    for r, h in rows:
        assert np.array_equal(part[r, h], full[r, h])


def test_decode_rows_helper_matches_full():
    wl = make_decode_case(24, [19, 70, 3], 8, 2, 64)
    full = A.paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    rows = [(0, 0), (1, 5), (2, 7), (1, 4)]
    part = A.paged_decode_rows(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, rows)
    for r in rows:
        assert np.array_equal(part[r], full[r])
