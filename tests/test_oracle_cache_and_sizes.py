"""Pins for the cache-write / block-copy oracle and the KV-size closed forms
(CPU only). Expected values come from tests/golden/*.txt, each line citing the
page that prints it."""
import math

import numpy as np
import pytest

from oracle import kv_sizes
from oracle.attention import gather_kv
from oracle.cache_ops import copy_blocks, reshape_and_cache, slot_to_block_offset
from tests.conftest import read_golden
from workloads import make_decode_case


# ------------------------------------------------------------ closed forms --

def test_kv_bytes_per_token_printed_values():
    rows = read_golden("kv_bytes_per_token.txt")
    assert len(rows) >= 7
    for L, H, D, dt, want in rows:
        assert kv_sizes.kv_bytes_per_token(int(L), int(H), int(D), int(dt)) == int(want)


def test_kv_cache_totals_printed_values():
    for L, H, D, dt, S, B, want in read_golden("kv_cache_totals.txt"):
        got = kv_sizes.kv_cache_bytes(int(L), int(H), int(D), int(dt), int(S), int(B)) / 1e9
        assert f"{got:.2f}" == want


def test_kv_calc_table_printed_values():
    models = [(32, 32, 128, 2), (32, 8, 128, 2), (80, 8, 128, 2), (60, 8, 128, 2)]
    for row in read_golden("kv_calc_table.txt"):
        ctx = int(row[0])
        for (L, H, D, dt), want in zip(models, row[1:]):
            got = kv_sizes.kv_bytes_per_token(L, H, D, dt) * ctx / 2 ** 30
            assert f"{got:.1f}GB" == want


def test_block_size_waste_printed_values():
    for bs, avg, want in read_golden("block_size_waste.txt"):
        got = kv_sizes.max_waste_fraction(int(bs), float(avg)) * 100
        assert f"{got:.1f}" == want


def test_tail_waste_bound():
    for n in range(1, 200):
        w = kv_sizes.tail_waste_slots(n, 16)
        assert 0 <= w <= 15
        assert (n + w) % 16 == 0


def test_decode_kv_read_bytes_matches_workload_sizes():
    # 7B-class MHA layer, 8 x 2048 tokens, 32 kv heads x 128 dims, bf16
    assert kv_sizes.decode_kv_read_bytes([2048] * 8, 32, 128) == 268_435_456
    # one layer of the 80-layer 70B model is 1/80 of the per-token closed form
    assert kv_sizes.decode_kv_read_bytes([1], 8, 128) * 80 == 327_680


# ------------------------------------------------------- block-table math --

def test_block_table_examples():
    rows = read_golden("block_table_examples.txt")
    table = None
    for r in rows:
        if r[0] == "table":
            table = [int(x) for x in r[1:]]
        elif r[0] == "range":
            first, last, blk = int(r[1]), int(r[2]), int(r[3])
            for t in range(first, last + 1):
                b, off = slot_to_block_offset(table[t // 16] * 16 + t % 16, 16)
                assert (b, off) == (blk, t - first)
        elif r[0] == "token":
            sep = r.index(";")
            tab = [int(x) for x in r[1:sep]]
            pos, blk, off = (int(x) for x in r[sep + 1:])
            b, o = slot_to_block_offset(tab[pos // 16] * 16 + pos % 16, 16)
            assert (b, o) == (blk, off)
        elif r[0] == "blocks":
            assert kv_sizes.blocks_for(int(r[1]), 16) == int(r[2])


def test_gather_follows_printed_table():
    """Put marker values in blocks 7, 2, 15, 3 and read them back in logical order."""
    pool = np.zeros((16, 1, 16, 2), np.float64)
    for i, blk in enumerate([7, 2, 15, 3]):
        for off in range(16):
            pool[blk, 0, off, :] = 16 * i + off
    got = gather_kv(pool, np.array([7, 2, 15, 3]), 64)
    assert np.array_equal(got[:, 0, 0], np.arange(64, dtype=np.float64))


# ---------------------------------------------------- reshape_and_cache --

def test_reshape_and_cache_scatter_round_trip():
    wl = make_decode_case(31, [6, 17, 32, 50], 4, 2, 64, n_new=5)
    kp, vp = reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    for b, n in enumerate(wl.dec_ctx):
        gk = gather_kv(kp, wl.dec_tables[b], int(n))
        gv = gather_kv(vp, wl.dec_tables[b], int(n))
        assert np.array_equal(gk, wl.seq_k[b])
        assert np.array_equal(gv, wl.seq_v[b])
    # exactly the slots named were written: every other uint16 is unchanged
    changed = np.argwhere((kp != wl.k_pool).any(axis=(1, 3)))
    written = {(int(s) // 16, int(s) % 16) for s in wl.slot_mapping}
    assert {(int(b), int(o)) for b, _, o in
            np.argwhere((kp != wl.k_pool).any(axis=3))} <= written
    assert len(changed) > 0


def test_reshape_and_cache_negative_slot_skips():
    wl = make_decode_case(32, [4, 4], 2, 2, 64, n_new=1)
    slots = wl.slot_mapping.copy()
    slots[1] = -1
    kp, vp = reshape_and_cache(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, slots)
    blk, off = divmod(int(wl.slot_mapping[1]), 16)
    assert np.array_equal(kp[blk, :, off], wl.k_pool[blk, :, off])
    blk0, off0 = divmod(int(slots[0]), 16)
    assert np.array_equal(kp[blk0, :, off0], wl.new_k[0])


def test_reshape_and_cache_bit_exact_including_nan_payloads():
    rng = np.random.default_rng(0)
    pool = rng.integers(0, 2 ** 16, size=(8, 2, 16, 64), dtype=np.uint16)
    new = rng.integers(0, 2 ** 16, size=(3, 2, 64), dtype=np.uint16)
    new[0, 0, :4] = [0x7FC1, 0xFFFF, 0x8000, 0x0001]   # NaN payloads, -0, denormal
    kp, _ = reshape_and_cache(new, new, pool, pool, np.array([5, 16 * 7 + 15, 33]))
    assert np.array_equal(kp[0, :, 5], new[0])
    assert np.array_equal(kp[7, :, 15], new[1])
    assert np.array_equal(kp[2, :, 1], new[2])


# ---------------------------------------------------------- copy_blocks --

def test_copy_blocks_copies_whole_block_and_nothing_else():
    rng = np.random.default_rng(1)
    kpool = rng.integers(0, 2 ** 16, size=(12, 4, 16, 64), dtype=np.uint16)
    vpool = rng.integers(0, 2 ** 16, size=(12, 4, 16, 64), dtype=np.uint16)
    pairs = np.array([[3, 9], [3, 10], [0, 11]], dtype=np.int64)
    kp, vp = copy_blocks(kpool, vpool, pairs)
    for s, d in pairs:
        assert np.array_equal(kp[d], kpool[s]) and np.array_equal(vp[d], vpool[s])
    untouched = [i for i in range(12) if i not in (9, 10, 11)]
    assert np.array_equal(kp[untouched], kpool[untouched])
    assert np.array_equal(vp[untouched], vpool[untouched])


def test_cow_copy_leaves_sibling_attention_unchanged():
    """After a shared block is copied and the copy overwritten, a sibling
    that still maps the original block sees the same K/V as before."""
    from oracle.attention import paged_decode
    wl = make_decode_case(33, [48, 48], 4, 4, 64, prefix_tokens=32, pool_factor=2.0)
    before = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    src = int(wl.dec_tables[1, 1])
    dst = int(wl.meta["perm_tail"][0])
    kp, vp = copy_blocks(wl.k_pool, wl.v_pool, np.array([[src, dst]]))
    tabs = wl.dec_tables.copy()
    tabs[1, 1] = dst
    same = paged_decode(wl.q, kp, vp, tabs, wl.dec_ctx, wl.scale)
    assert np.array_equal(same, before)           # a copy changes nothing
    kp2, vp2 = reshape_and_cache(np.full((1, 4, 64), 0x3F80, np.uint16),
                                 np.full((1, 4, 64), 0x4000, np.uint16),
                                 kp, vp, np.array([dst * 16 + 3]))
    after = paged_decode(wl.q, kp2, vp2, tabs, wl.dec_ctx, wl.scale)
    assert np.array_equal(after[0], before[0])     # sibling unchanged
    assert not np.array_equal(after[1], before[1])  # the diverged sequence changed


def test_swap_round_trip_moves_blocks_to_new_places():
    from oracle.cache_ops import swap_in, swap_out
    from workloads import make_decode_case
    wl = make_decode_case(91, [40, 70], 8, 2, 64, num_blocks=40, n_new=0)
    ids = list(wl.dec_tables[1, :5])
    hk, hv = swap_out(wl.k_pool, wl.v_pool, ids)
    for i, b in enumerate(ids):
        assert np.array_equal(hk[i], wl.k_pool[b]) and np.array_equal(hv[i], wl.v_pool[b])
    free = [b for b in range(wl.num_blocks) if b not in set(wl.dec_tables.ravel())][:5]
    kp, vp = swap_in(hk, hv, wl.k_pool, wl.v_pool, free)
    for i, b in enumerate(free):
        assert np.array_equal(kp[b], wl.k_pool[ids[i]]) and np.array_equal(vp[b], wl.v_pool[ids[i]])
    untouched = [b for b in range(wl.num_blocks) if b not in set(free)]
    assert np.array_equal(kp[untouched], wl.k_pool[untouched])
    # decode over the moved blocks equals decode over the originals (paging is addressing only)
    from oracle.attention import paged_decode
    t2 = wl.dec_tables.copy()
    t2[1, :5] = free
    a = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    b = paged_decode(wl.q, kp, vp, t2, wl.dec_ctx, wl.scale)
    assert np.array_equal(a, b)
