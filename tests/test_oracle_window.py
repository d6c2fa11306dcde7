"""Pins for sliding-window decode and window-driven block release (CPU).

The windowed oracle is tied to the full-context oracle (a window that
reaches position 0), to a closed form (window 0 returns the newest V row),
to torch SDPA with an explicit band mask over the logical, never-paged K/V,
and the block release to the refcount invariants.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode, paged_decode_window
from oracle.bf16 import bf16_bits_to_f64
from oracle.block_manager import BlockManagerError, BlockManagerModel
from workloads import BF16_NAN, make_decode_case, make_decode_case_window

torch = pytest.importorskip("torch")


def _released_copy(wl, window):
    """The same batch with every block wholly before each window released:
    table entry -1 and the block's content poisoned with NaN."""
    tabs = wl.dec_tables.copy()
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    for b, n in enumerate(wl.dec_ctx):
        first = max(0, int(n) - 1 - window)
        for j in range(first // 16):
            kp[tabs[b, j]] = BF16_NAN
            vp[tabs[b, j]] = BF16_NAN
            tabs[b, j] = -1
    return tabs, kp, vp


@pytest.mark.parametrize("window", [0, 1, 15, 16, 17, 40])
def test_window_matches_sdpa_band_mask(window):
    wl = make_decode_case(51, [1, 2, 16, 17, 33, 64, 100], 8, 2, 64, n_new=0, keep_logical=True)
    tabs, kp, vp = _released_copy(wl, window)
    got = paged_decode_window(wl.q, kp, vp, tabs, wl.dec_ctx, wl.scale, window)
    F = torch.nn.functional
    for b, n in enumerate(wl.dec_ctx):
        n = int(n)
        k = torch.from_numpy(bf16_bits_to_f64(wl.seq_k[b]).transpose(1, 0, 2).copy())[None]  # [1][Hk][n][D]
        v = torch.from_numpy(bf16_bits_to_f64(wl.seq_v[b]).transpose(1, 0, 2).copy())[None]
        q = torch.from_numpy(bf16_bits_to_f64(wl.q[b]))[None, :, None, :]                 # [1][H][1][D]
        pos = torch.arange(n)
        mask = (pos >= n - 1 - window) & (pos <= n - 1)                                    # band [i-W, i]
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask[None, None, None, :], scale=wl.scale,
                                             enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-11, atol=1e-12)
    assert np.isfinite(got).all()


def test_window_covering_everything_is_full_attention():
    wl = make_decode_case(52, [1, 15, 16, 37, 300], 8, 2, 64, n_new=0)
    full = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    for window in (299, 300, 10 ** 6):
        got = paged_decode_window(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, window)
        assert np.array_equal(got, full)


def test_window_zero_returns_newest_v():
    wl = make_decode_case(53, [1, 9, 16, 17, 50], 8, 4, 64, n_new=0, keep_logical=True)
    got = paged_decode_window(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, 0)
    for b, n in enumerate(wl.dec_ctx):
        v_last = bf16_bits_to_f64(wl.seq_v[b][int(n) - 1])     # [Hk][D]
        for h in range(8):
            assert np.array_equal(got[b, h], v_last[h // 2])


def test_generator_holds_exactly_the_window_blocks():
    wl = make_decode_case_window(54, [1, 16, 17, 40, 100, 300], 4, 2, 64, window=20)
    for b, n in enumerate(wl.dec_ctx):
        first_blk = max(0, int(n) - 1 - 20) // 16
        row = wl.dec_tables[b]
        assert (row[:first_blk] == -1).all()
        assert (row[first_blk:(int(n) + 15) // 16] >= 0).all()


# ------------------------------------------------------------ block release

def test_release_before_frees_whole_blocks_only():
    m = BlockManagerModel(32, 16)
    m.add_seq(0)
    m.append_tokens(0, 70)                       # blocks 0..4, last holds 6 tokens
    t = m.block_table(0)
    dropped = m.release_before(0, 47)            # blocks wholly before 47: 0, 1
    assert dropped == t[:2]
    assert m.block_table(0)[:2] == [-1, -1] and m.block_table(0)[2:] == t[2:]
    assert m.num_free() == 32 - 3
    assert m.release_before(0, 47) == []         # idempotent
    m.check_invariants()
    slots, _ = m.append_tokens(0, 30)            # appends continue at the end
    assert all(s // 16 not in (t[0], t[1]) or s // 16 in m.block_table(0) for s in slots)
    m.check_invariants()


def test_release_of_shared_blocks_decrefs():
    m = BlockManagerModel(16, 16)
    m.add_seq(0)
    m.append_tokens(0, 48)
    m.fork(0, 1)
    t = m.block_table(0)
    assert [m.refcount(b) for b in t] == [2, 2, 2]
    m.release_before(1, 40)                      # the child drops blocks 0, 1
    assert [m.refcount(b) for b in t] == [1, 1, 2]
    assert m.num_free() == 16 - 3                # still held by the parent
    m.release_before(0, 40)
    assert m.num_free() == 16 - 1
    m.fork(1, 2)                                 # holes are not incref'd
    assert m.refcount(t[2]) == 3
    m.check_invariants()
    for s in (0, 1, 2):
        m.free_seq(s)
    assert m.num_free() == 16
    m.check_invariants()


def test_released_block_cannot_be_made_private():
    m = BlockManagerModel(8, 16)
    m.add_seq(0)
    m.append_tokens(0, 40)
    m.release_before(0, 32)
    with pytest.raises(BlockManagerError):
        m.make_private(0, 0)


def test_random_windowed_appends_keep_the_pool_bounded():
    """Appending with a release after every step keeps at most
    ceil((W + 1) / 16) + 1 blocks per sequence (the cache is O(W))."""
    rng = np.random.default_rng(9)
    W = 40
    m = BlockManagerModel(64, 16)
    for s in range(4):
        m.add_seq(s)
    for _ in range(400):
        s = int(rng.integers(0, 4))
        m.append_tokens(s, 1)
        n = m.seq_len(s)
        m.release_before(s, max(0, n - 1 - W))
        held = sum(1 for b in m.block_table(s) if b >= 0)
        assert held <= (W + 1 + 15) // 16 + 1
        m.check_invariants()
