"""GPU parity: reshape_and_cache and copy_blocks must match the oracle bit for
bit (they are copies)."""
import numpy as np
import pytest

from oracle.cache_ops import copy_blocks as o_copy
from oracle.cache_ops import reshape_and_cache as o_rac
from tests._gpu import check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


@pytest.mark.parametrize("D,Hk,n_new", [(64, 2, 5), (128, 8, 1), (128, 1, 3), (64, 16, 2)])
def test_reshape_and_cache_bit_exact(pk, D, Hk, n_new):
    wl = make_decode_case(40 + D + Hk, [5, 16, 17, 33, 70], 2 * Hk, Hk, D, n_new=n_new)
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    assert np.array_equal(host_bits(kp), ek)
    assert np.array_equal(host_bits(vp), ev)
    check_device_error(0)


def test_reshape_and_cache_skips_negative_and_flags_out_of_range(pk):
    wl = make_decode_case(50, [8, 9, 10], 4, 4, 64, n_new=1)
    slots = wl.slot_mapping.copy()
    slots[0] = -1
    slots[2] = wl.num_blocks * 16 + 3          # outside the pool
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(slots))
    keep = slots.copy()
    keep[2] = -1                                 # the oracle writes neither row
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, keep)
    assert np.array_equal(host_bits(kp), ek) and np.array_equal(host_bits(vp), ev)
    check_device_error(2)                        # PA_DEVERR_SLOT


def test_reshape_and_cache_full_mixed_step(pk):
    """Config-sized scatter: 60 decode tokens + 4 x 512 chunk tokens."""
    wl = make_workload("mixed", fill="nan", keep_logical=False)
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    blocks = np.unique(wl.slot_mapping // 16)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool[blocks], wl.v_pool[blocks],
                   np.searchsorted(blocks, wl.slot_mapping // 16) * 16 + wl.slot_mapping % 16)
    gk = host_bits(kp)[blocks]
    gv = host_bits(vp)[blocks]
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)
    check_device_error(0)


@pytest.mark.parametrize("D,Hk", [(64, 2), (128, 8)])
def test_copy_blocks_bit_exact(pk, D, Hk):
    rng = np.random.default_rng(D + Hk)
    nb = 40
    kpool = rng.integers(0, 2 ** 16, size=(nb, Hk, 16, D), dtype=np.uint16)
    vpool = rng.integers(0, 2 ** 16, size=(nb, Hk, 16, D), dtype=np.uint16)
    pairs = np.array([[3, 30], [3, 31], [7, 32], [39, 0]], dtype=np.int64)
    kp, vp = dev(kpool), dev(vpool)
    pk.pa_copy_blocks(kp, vp, dev(pairs))
    ek, ev = o_copy(kpool, vpool, pairs)
    assert np.array_equal(host_bits(kp), ek) and np.array_equal(host_bits(vp), ev)
    check_device_error(0)


def test_copy_blocks_flags_bad_pair(pk):
    kpool = np.arange(8 * 2 * 16 * 64, dtype=np.uint16).reshape(8, 2, 16, 64)
    pairs = np.array([[1, 2], [5, 8], [-1, 3]], dtype=np.int64)
    kp, vp = dev(kpool), dev(kpool)
    pk.pa_copy_blocks(kp, vp, dev(pairs))
    ek, _ = o_copy(kpool, kpool, pairs[:1])
    assert np.array_equal(host_bits(kp), ek)
    check_device_error(8)                        # PA_DEVERR_PAIR


@pytest.mark.parametrize("D,Hk", [(64, 8), (128, 8), (128, 2)])
def test_copy_blocks_fp8_pool_bit_exact(pk, D, Hk):
    """Copy-on-write in an E4M3 pool (1-byte elements): the block size in
    bytes is half the bf16 one, so a copy sized for bf16 would move the wrong
    bytes and, for a destination in the upper half of the pool, write past its
    end. Destinations here sit in the upper half and at the last block."""
    torch = torch_cuda()
    rng = np.random.default_rng(700 + D + Hk)
    nb = 48
    kpool = rng.integers(0, 256, size=(nb, Hk, 16, D), dtype=np.uint8)
    vpool = rng.integers(0, 256, size=(nb, Hk, 16, D), dtype=np.uint8)
    pairs = np.array([[3, 30], [3, 47], [7, 40], [39, 0], [12, 25]], dtype=np.int64)
    # guard bytes after each pool catch a copy that runs past the end
    guard = 4096
    kbuf = torch.full((nb * Hk * 16 * D + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    vbuf = torch.full((nb * Hk * 16 * D + guard,), 0x5A, dtype=torch.uint8, device="cuda")
    kp = kbuf[: nb * Hk * 16 * D].view(nb, Hk, 16, D)
    vp = vbuf[: nb * Hk * 16 * D].view(nb, Hk, 16, D)
    kp.copy_(torch.from_numpy(kpool))
    vp.copy_(torch.from_numpy(vpool))
    pk.pa_copy_blocks(kp, vp, dev(pairs))
    ek, ev = o_copy(kpool, vpool, pairs)
    assert np.array_equal(kp.cpu().numpy(), ek)
    assert np.array_equal(vp.cpu().numpy(), ev)
    assert bool((kbuf[nb * Hk * 16 * D:] == 0xA5).all()) and bool((vbuf[nb * Hk * 16 * D:] == 0x5A).all())
    check_device_error(0)


def test_copy_blocks_fp8_flags_bad_pair(pk):
    kpool = (np.arange(8 * 2 * 16 * 64) % 251).astype(np.uint8).reshape(8, 2, 16, 64)
    pairs = np.array([[1, 2], [5, 8], [-1, 3]], dtype=np.int64)
    kp, vp = dev(kpool), dev(kpool.copy())
    pk.pa_copy_blocks(kp, vp, dev(pairs))
    ek, _ = o_copy(kpool, kpool, pairs[:1])
    assert np.array_equal(kp.cpu().numpy(), ek)
    check_device_error(8)                        # PA_DEVERR_PAIR
