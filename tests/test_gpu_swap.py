"""GPU parity for swapping blocks between the pools and page-locked host
memory (preemption), and the whole preemption flow through the C++ block
manager: bit-exact against the oracle's gather / scatter, and decode after a
swap-out, reuse of the freed blocks by another sequence and a swap-in into
new blocks equal, bit for bit, to decode before it.
"""
import numpy as np
import pytest

from oracle.cache_ops import swap_in as o_swap_in
from oracle.cache_ops import swap_out as o_swap_out
from tests._gpu import check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_decode_case_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def _pinned_like(shape, dtype):
    torch = torch_cuda()
    return torch.empty(shape, dtype=dtype).pin_memory()


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_swap_out_and_in_bit_exact(pk, kind):
    torch = torch_cuda()
    if kind == "bf16":
        wl = make_decode_case(700, [40, 300, 129], 32, 8, 128, num_blocks=80, n_new=0)
        tdt = torch.int16
    else:
        wl = make_decode_case_fp8(701, [40, 300, 129], 32, 8, 128, num_blocks=80, n_new=0)
        tdt = torch.uint8
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    ids = np.array(list(wl.dec_tables[1, :19]) + [int(wl.dec_tables[0, 2])], dtype=np.int32)
    hk = _pinned_like((len(ids),) + wl.k_pool.shape[1:], tdt)
    hv = _pinned_like((len(ids),) + wl.v_pool.shape[1:], tdt)
    pk.pa_swap_out_blocks(kp, vp, dev(ids), hk, hv)
    torch.cuda.synchronize()
    ek, ev = o_swap_out(wl.k_pool, wl.v_pool, ids)
    view = np.uint16 if kind == "bf16" else np.uint8
    assert np.array_equal(hk.numpy().view(view), ek) and np.array_equal(hv.numpy().view(view), ev)
    # swap in to different blocks (unused by any table)
    used = set(int(b) for b in wl.dec_tables.ravel() if b >= 0)
    dst = np.array([b for b in range(wl.num_blocks) if b not in used][:len(ids)], dtype=np.int32)
    pk.pa_swap_in_blocks(hk, hv, kp, vp, dev(dst))
    torch.cuda.synchronize()
    xk, xv = o_swap_in(ek, ev, wl.k_pool, wl.v_pool, dst)
    assert np.array_equal(kp.cpu().numpy().view(view), xk) and np.array_equal(vp.cpu().numpy().view(view), xv)
    check_device_error(0)


def test_swap_bad_block_id_sets_flag_and_skips(pk):
    torch = torch_cuda()
    wl = make_decode_case(702, [40], 8, 2, 64, num_blocks=8, n_new=0)
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    ids = np.array([1, 99, 2], dtype=np.int32)
    hk = torch.zeros((3,) + wl.k_pool.shape[1:], dtype=torch.int16).pin_memory()
    hv = torch.zeros((3,) + wl.v_pool.shape[1:], dtype=torch.int16).pin_memory()
    pk.pa_swap_out_blocks(kp, vp, dev(ids), hk, hv)
    torch.cuda.synchronize()
    check_device_error(1)  # PA_DEVERR_BLOCK_ID
    got = hk.numpy().view(np.uint16)
    assert np.array_equal(got[0], wl.k_pool[1]) and np.array_equal(got[2], wl.k_pool[2])
    assert (got[1] == 0).all()


def test_preemption_flow_decodes_identically(pk):
    """Three sequences share nothing; sequence 1 is preempted (swap-out of its
    private tail), sequence 2 grows into the freed blocks (new K/V written
    there), sequence 1 is swapped back into fresh blocks: its decode output is
    bit-identical to the one before preemption."""
    torch = torch_cuda()
    rng = np.random.default_rng(5)
    H, Hk, D, NB = 32, 8, 128, 96
    bm = pk.BlockManager(NB, 16)
    kp = torch.zeros((NB, Hk, 16, D), dtype=torch.int16, device="cuda")
    vp = torch.zeros_like(kp)

    def write(seq, n):
        slots, _ = bm.append_tokens(seq, n)
        kv = lambda: torch.from_numpy(rng.standard_normal((n, Hk, D), dtype=np.float32)).to(torch.bfloat16) \
            .view(torch.int16).cuda()
        pk.pa_reshape_and_cache(kv(), kv(), kp, vp, torch.tensor(slots, dtype=torch.int64, device="cuda"))

    for s, n in ((0, 300), (1, 517), (2, 64)):
        bm.add_seq(s)
        write(s, n)
    q = torch.from_numpy(rng.standard_normal((3, H, D), dtype=np.float32)).to(torch.bfloat16).view(torch.int16).cuda()

    def decode():
        tabs, ctx = bm.build_batch([0, 1, 2], 48)
        out = torch.empty_like(q)
        ws = pk.decode_workspace(q, 768)
        pk.pa_decode(out, q, kp, vp, dev(tabs), dev(ctx), 0.0883883, 768, workspace=ws)
        torch.cuda.synchronize()
        return host_bits(out)

    before = decode()
    out_ids = bm.swap_out(1)
    assert len(out_ids) == 33                        # 517 tokens: all 33 blocks are private
    hk = torch.empty((len(out_ids), Hk, 16, D), dtype=torch.int16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pk.pa_swap_out_blocks(kp, vp, dev(np.array(out_ids, np.int32)), hk, hv)
    write(2, 600)                                    # takes (and overwrites) freed blocks
    in_ids = bm.swap_in(1)
    assert len(in_ids) == 33 and in_ids != out_ids
    pk.pa_swap_in_blocks(hk, hv, kp, vp, dev(np.array(in_ids, np.int32)))
    after = decode()
    assert np.array_equal(after[1], before[1])
    assert np.array_equal(after[0], before[0])
    check_device_error(0)
