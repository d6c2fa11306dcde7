"""C ABI checks that need no GPU: the library loads, exports every function
the header declares, validates arguments before touching the device, and the
host block manager matches the reference model."""
import ctypes as C
import os
import random
import re

import numpy as np
import pytest

from oracle.block_manager import BlockManagerError, BlockManagerModel, OutOfBlocks
from tests.conftest import ROOT


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for must in ["pa_decode", "pa_decode_ex", "pa_decode_workspace_bytes", "pa_reshape_and_cache",
                 "pa_copy_blocks", "pa_prefill_paged", "pa_get_device_error", "pa_status_string",
                 "pa_bm_create", "pa_bm_append_tokens", "pa_bm_fork", "pa_bm_free_seq"]:
        assert must in names


def test_library_exports_every_declared_symbol(capi):
    from paged_kv_cache_59_gb300 import _capi
    for name in _declared_functions():
        assert hasattr(capi, name), name
        assert name in _capi.SIGNATURES, f"binding lacks {name}"


def test_status_strings(capi):
    assert capi.pa_status_string(0) == b"ok"
    assert b"unsupported" in capi.pa_status_string(-2)


def test_workspace_size_formula(capi):
    # 64 seqs x 32 heads, context up to 4096, 512-token partitions -> 8 partitions
    rows = 64 * 32 * 8
    ml = (rows * 8 + 255) // 256 * 256
    assert capi.pa_decode_workspace_bytes(64, 32, 128, 4096, 512) == ml + rows * 128 * 4
    assert capi.pa_decode_workspace_bytes(4, 4, 64, 37, 512) == 0      # one partition
    assert capi.pa_decode_workspace_bytes(4, 4, 64, 37, 100) == 0      # invalid size -> 0


def _decode_args(**over):
    a = dict(out=C.c_void_p(16), q=C.c_void_p(32), k=C.c_void_p(64), v=C.c_void_p(128),
             tab=C.c_void_p(256), ctx=C.c_void_p(512), scale=0.125, H=4, Hk=4, D=64, bs=16,
             B=4, maxb=4, maxctx=64, nblk=32, pt=0, ws=C.c_void_p(None), wsb=0, stream=None)
    a.update(over)
    return a


def _call_decode(capi, a):
    return capi.pa_decode_ex(a["out"], a["q"], a["k"], a["v"], a["tab"], a["ctx"], a["scale"],
                             a["H"], a["Hk"], a["D"], a["bs"], a["B"], a["maxb"], a["maxctx"],
                             a["nblk"], a["pt"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(D=96), -2), (dict(bs=32), -2), (dict(H=6, Hk=4), -1), (dict(H=48, Hk=3), -2),
    (dict(B=-1), -1), (dict(maxb=2), -1), (dict(pt=100), -1), (dict(pt=4096), -1),
    (dict(q=C.c_void_p(33)), -1), (dict(out=C.c_void_p(32)), -1), (dict(k=C.c_void_p(None)), -1),
    (dict(maxctx=1000, maxb=100), -3),
])
def test_decode_argument_errors_need_no_device(capi, over, status):
    assert _call_decode(capi, _decode_args(**over)) == status


def test_decode_empty_batch_is_ok(capi):
    assert _call_decode(capi, _decode_args(B=0)) == 0


def test_cache_ops_argument_errors(capi):
    p = C.c_void_p(64)
    assert capi.pa_reshape_and_cache(p, p, p, p, p, 4, 2, 64, 8, 16, None) == -2
    assert capi.pa_reshape_and_cache(p, p, p, p, p, -1, 2, 64, 16, 16, None) == -1
    assert capi.pa_reshape_and_cache(p, p, p, p, p, 0, 2, 64, 16, 16, None) == 0
    assert capi.pa_reshape_and_cache(C.c_void_p(8), p, p, p, p, 4, 2, 64, 16, 16, None) == -1
    assert capi.pa_copy_blocks(p, p, p, 3, 2, 64, 4, 16, None) == -2
    assert capi.pa_copy_blocks(p, p, p, 0, 2, 64, 16, 16, None) == 0
    assert capi.pa_copy_blocks(p, p, C.c_void_p(12), 3, 2, 64, 16, 16, None) == -1
    # element size: 1 (fp8) and 2 (bf16) only
    for eb in (0, 3, 4, -1):
        assert capi.pa_copy_blocks_ex(p, p, p, 3, 2, 64, 16, eb, 16, None) == -1
    assert capi.pa_copy_blocks_ex(p, p, p, 0, 2, 64, 16, 1, 16, None) == 0
    assert capi.pa_copy_blocks_ex(p, p, p, 3, 2, 64, 4, 1, 16, None) == -2
    assert capi.pa_copy_blocks_ex(C.c_void_p(72), p, p, 3, 2, 64, 16, 1, 16, None) == -1


def test_fp8_argument_errors_need_no_device(capi):
    p = C.c_void_p(4096)
    # cache write: block size 8, head_dim 60, missing scale, misaligned k, empty
    assert capi.pa_reshape_and_cache_fp8(p, p, p, p, p, p, p, 4, 2, 64, 8, 16, None) == -2
    assert capi.pa_reshape_and_cache_fp8(p, p, p, p, p, p, p, 4, 2, 60, 16, 16, None) == -2
    assert capi.pa_reshape_and_cache_fp8(p, p, p, p, p, None, p, 4, 2, 64, 16, 16, None) == -1
    assert capi.pa_reshape_and_cache_fp8(C.c_void_p(4104), p, p, p, p, p, p, 4, 2, 64, 16, 16, None) == -1
    assert capi.pa_reshape_and_cache_fp8(p, p, p, p, p, p, p, 0, 2, 64, 16, 16, None) == 0
    # decode: missing or misaligned scales, unsupported head_dim, group 3, empty batch
    tail = [C.c_float(0.1), 8, 2, 128, 16, 4, 64, 1024, 256, 0, None, 0, None]
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, None, p, p, p, *tail) == -1
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, p, C.c_void_p(4098), p, p, *tail) == -1
    bad_d = list(tail); bad_d[3] = 96
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, p, p, p, p, *bad_d) == -2
    bad_g = list(tail); bad_g[1], bad_g[2] = 6, 2
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, p, p, p, p, *bad_g) == -2
    empty = list(tail); empty[5] = 0
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, p, p, p, p, *empty) == 0
    # a batch that needs split-K scratch and gets none (contexts up to 2048 tokens: two of the
    # tensor-core kernel's default 1024-token partitions)
    big = list(tail); big[6], big[7] = 128, 2048
    assert capi.pa_decode_fp8(p, C.c_void_p(8192), p, p, p, p, p, p, *big) == -3


# ----------------------------------------------------------- block manager --

def test_block_manager_matches_model_on_random_operations(capi):
    from paged_kv_cache_59_gb300 import BlockManager, PagedKVError
    rng = random.Random(7)
    for trial in range(25):
        nb = rng.randint(3, 48)
        model = BlockManagerModel(nb, 16)
        bm = BlockManager(nb, 16)
        live, next_id = [], 0
        for _ in range(250):
            op = rng.random()
            if op < 0.2 or not live:
                model.add_seq(next_id); bm.add_seq(next_id); live.append(next_id); next_id += 1
            elif op < 0.6:
                s, n = rng.choice(live), rng.randint(0, 40)
                try:
                    want = model.append_tokens(s, n)
                except OutOfBlocks:
                    with pytest.raises(PagedKVError) as e:
                        bm.append_tokens(s, n)
                    assert e.value.status == -6
                else:
                    assert bm.append_tokens(s, n) == want
            elif op < 0.72:
                model.fork(live[0], next_id); bm.fork(live[0], next_id)
                live.append(next_id); next_id += 1
            elif op < 0.82:
                s = rng.choice(live)
                if model.block_table(s):
                    lb = rng.randrange(len(model.block_table(s)))
                    try:
                        want = model.make_private(s, lb)
                    except OutOfBlocks:
                        with pytest.raises(PagedKVError):
                            bm.make_private(s, lb)
                    except BlockManagerError:          # a block released by the window
                        with pytest.raises(PagedKVError) as e:
                            bm.make_private(s, lb)
                        assert e.value.status == -1
                    else:
                        assert bm.make_private(s, lb) == want
            elif op < 0.9:
                s = rng.choice(live)
                first = rng.randint(0, model.seq_len(s) + 5)
                assert bm.release_before(s, first) == len(model.release_before(s, first))
            else:
                s = rng.choice(live)
                model.free_seq(s); bm.free_seq(s); live.remove(s)
            model.check_invariants()
            assert bm.num_free() == model.num_free()
            for s in live:
                assert bm.block_table(s) == model.block_table(s)
                assert bm.seq_len(s) == model.seq_len(s)
            for b in range(nb):
                assert bm.refcount(b) == model.refcount(b)


def test_block_manager_errors_and_batch_tables(capi):
    from paged_kv_cache_59_gb300 import BlockManager, PagedKVError
    bm = BlockManager(8, 16)
    bm.add_seq(1)
    with pytest.raises(PagedKVError):
        bm.add_seq(1)
    with pytest.raises(PagedKVError):
        bm.free_seq(2)
    with pytest.raises(PagedKVError):
        bm.fork(5, 6)
    bm.append_tokens(1, 40)
    bm.add_seq(2)
    bm.append_tokens(2, 3)
    tabs, lens = bm.build_batch([1, 2], 4)
    assert list(lens) == [40, 3]
    assert list(tabs[0][:3]) == bm.block_table(1) and tabs[0][3] == -1
    assert list(tabs[1][:1]) == bm.block_table(2) and list(tabs[1][1:]) == [-1, -1, -1]
    with pytest.raises(PagedKVError):
        bm.build_batch([1], 2)
    assert bm.refcount(0) >= 0
    with pytest.raises(PagedKVError):
        bm.refcount(8)


def test_prefix_cache_matches_model_on_random_operations(capi):
    """The C++ manager's prefix cache against the model: admissions that reuse
    cached prefixes, appends, cache registrations, forks, window releases,
    copies and frees, with eviction under a small pool; tables, refcounts,
    free and cached counts compared after every operation."""
    from paged_kv_cache_59_gb300 import BlockManager, PagedKVError
    rng = random.Random(23)
    for trial in range(12):
        nb = rng.randint(6, 60)
        model, bm = BlockManagerModel(nb, 16), BlockManager(nb, 16)
        prompts = [[rng.randrange(30) for _ in range(rng.randrange(1, 120))] for _ in range(6)]
        toks, nxt = {}, 0
        for _ in range(300):
            op = rng.random()
            if op < 0.35:
                t = list(rng.choice(prompts)) + [rng.randrange(30) for _ in range(rng.randrange(0, 25))]
                got = model.add_seq_cached(nxt, t)
                assert bm.add_seq_cached(nxt, t) == got
                toks[nxt] = t
                try:
                    want = model.append_tokens(nxt, len(t) - got)
                except OutOfBlocks:
                    with pytest.raises(PagedKVError) as e:
                        bm.append_tokens(nxt, len(t) - got)
                    assert e.value.status == -6
                    model.free_seq(nxt); bm.free_seq(nxt); del toks[nxt]
                else:
                    assert bm.append_tokens(nxt, len(t) - got) == want
                    assert bm.cache_blocks(nxt, t) == model.cache_full_blocks(nxt, t)
                nxt += 1
            elif op < 0.5 and toks:
                s_ = rng.choice(list(toks))
                if s_ in model.swapped:
                    with pytest.raises(PagedKVError) as e:
                        bm.append_tokens(s_, 1)
                    assert e.value.status == -1
                    continue
                extra = [rng.randrange(30) for _ in range(rng.randrange(1, 30))]
                try:
                    want = model.append_tokens(s_, len(extra))
                except OutOfBlocks:
                    with pytest.raises(PagedKVError):
                        bm.append_tokens(s_, len(extra))
                else:
                    assert bm.append_tokens(s_, len(extra)) == want
                    toks[s_] = toks[s_] + extra
                    assert bm.cache_blocks(s_, toks[s_]) == model.cache_full_blocks(s_, toks[s_])
            elif op < 0.58 and toks:
                s_ = rng.choice(list(toks))
                if s_ in model.swapped:
                    continue
                model.fork(s_, nxt); bm.fork(s_, nxt)
                toks[nxt] = list(toks[s_]); nxt += 1
            elif op < 0.66 and toks:
                s_ = rng.choice(list(toks))
                if s_ in model.swapped:
                    continue
                first = rng.randint(0, model.seq_len(s_))
                assert bm.release_before(s_, first) == len(model.release_before(s_, first))
            elif op < 0.74 and toks:
                s_ = rng.choice(list(toks))
                if s_ in model.swapped:
                    continue
                if model.block_table(s_):
                    lb = rng.randrange(len(model.block_table(s_)))
                    try:
                        want = model.make_private(s_, lb)
                    except (OutOfBlocks, BlockManagerError):
                        with pytest.raises(PagedKVError):
                            bm.make_private(s_, lb)
                    else:
                        assert bm.make_private(s_, lb) == want
            elif op < 0.84 and toks:
                s_ = rng.choice(list(toks))
                if s_ in model.swapped:
                    try:
                        want = model.swap_in(s_)
                    except OutOfBlocks:
                        with pytest.raises(PagedKVError) as e:
                            bm.swap_in(s_)
                        assert e.value.status == -6
                    else:
                        assert len(bm.swap_in(s_)) == len(want)
                else:
                    assert len(bm.swap_out(s_)) == len(model.swap_out(s_))
            elif toks:
                s_ = rng.choice(list(toks))
                model.free_seq(s_); bm.free_seq(s_); del toks[s_]
            model.check_invariants()
            assert bm.num_free() == model.num_free()
            assert bm.num_cached() == model.num_cached()
            for s_ in toks:
                assert bm.block_table(s_) == model.block_table(s_)
                assert bm.seq_len(s_) == model.seq_len(s_)
            for b in range(nb):
                assert bm.refcount(b) == model.refcount(b)


def test_prefill_workspace_formula_and_errors(capi):
    # pieces of partials: pairs per sequence x kv heads x sequences x splits x 2 tiles x 128 rows x 132 floats
    pairs = (512 + 63) // 64                     # G = 4: 32 tokens per tile, 64 per pair
    assert capi.pa_prefill_workspace_bytes(4, 32, 8, 512, 3) == pairs * 8 * 4 * 3 * 2 * 128 * 132 * 4
    assert capi.pa_prefill_workspace_bytes(4, 32, 8, 512, 1) == 0
    assert capi.pa_prefill_workspace_bytes(4, 32, 6, 512, 2) == 0   # group 32/6: not supported
    assert capi.pa_prefill_workspace_bytes(0, 32, 8, 512, 2) == 0
    assert capi.pa_prefill_workspace_bytes(4, 32, 8, 512, 65) == 0
    # balanced (splits 0): 4 partial slots per SM, the work list (items + 4 per SM, 16 bytes each)
    # and 16 bytes of counters; 0 with no device
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 0
    items = pairs * 8 * 4
    want = (4 * sms * 2 * 128 * 132 * 4 + (items + 4 * sms) * 16 + 16) if sms else 0
    assert capi.pa_prefill_workspace_bytes(4, 32, 8, 512, 0) == want
    p = C.c_void_p(4096)
    args = [C.c_void_p(8192), p, p, p, p, p, p, C.c_float(0.1), 32, 8, 128, 16, 2, 4, 512, 16]
    assert capi.pa_prefill_paged_ex(*args, 3, None, 0, None) == -3      # split needs a workspace
    assert capi.pa_prefill_paged_ex(*args, -1, None, 0, None) == -1
    assert capi.pa_prefill_paged_ex(*args, 65, None, 0, None) == -1


def test_prefill_argument_errors_need_no_device(capi):
    p = C.c_void_p(4096)
    args = [p, p, p, p, p, p, p, C.c_float(0.1)]
    # head_dim 96 is not built for prefill (64 and 128 are); block size 8 unsupported; group 3 unsupported
    assert capi.pa_prefill_paged(*args, 8, 8, 96, 16, 2, 4, 64, 16, None) == -2
    assert capi.pa_prefill_paged(*args, 8, 8, 128, 8, 2, 4, 64, 16, None) == -2
    assert capi.pa_prefill_paged(*args, 12, 4, 128, 16, 2, 4, 64, 16, None) == -2
    assert capi.pa_prefill_paged(*args, 8, 8, 128, 16, -1, 4, 64, 16, None) == -1
    assert capi.pa_prefill_paged(*args, 8, 8, 128, 16, 0, 4, 64, 16, None) == 0
    assert capi.pa_prefill_paged(C.c_void_p(4100), *args[1:], 8, 8, 128, 16, 2, 4, 64, 16, None) == -1


def test_decode_tc_unsupported_shapes_need_no_device(capi):
    p = C.c_void_p(4096)
    args = [p, p, p, p, p, p, C.c_float(0.1)]
    # head_dim 64 has no tensor-core kernel; a pool too large for int32 TMA rows
    assert capi.pa_decode_tc(*args, 8, 8, 64, 16, 2, 4, 64, 16, 0, None, 0, None) == -2
    assert capi.pa_decode_tc(*args, 8, 8, 128, 16, 2, 4, 64, 20000000, 0, None, 0, None) == -2
    assert capi.pa_decode_tc(*args, 8, 8, 128, 16, 0, 4, 64, 16, 0, None, 0, None) == 0   # no sequences


def test_binding_refuses_host_tensors(capi):
    """No CPU fallback: every compute entry point of the binding rejects host
    tensors before anything reaches the library."""
    import torch
    import paged_kv_cache_59_gb300 as pk
    n, H, Hk, D, nb = 2, 8, 2, 64, 4
    q = torch.zeros(n, H, D, dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    kp = torch.zeros(nb, Hk, 16, D, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    tabs = torch.zeros(n, 2, dtype=torch.int32)
    ctx = torch.ones(n, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pk.pa_decode(out, q, kp, vp, tabs, ctx, 0.125, 1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pk.pa_decode_window(out, q, kp, vp, tabs, ctx, 0.125, 1, 4)
    k_new = torch.zeros(n, Hk, D, dtype=torch.bfloat16)
    slots = torch.zeros(n, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pk.pa_reshape_and_cache(k_new, k_new, kp, vp, slots)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pk.pa_copy_blocks(kp, vp, torch.zeros(1, 2, dtype=torch.int64))


@pytest.mark.parametrize("H,Hk,D", [(32, 8, 128), (64, 8, 128), (8, 8, 64), (16, 2, 64), (8, 1, 128)])
@pytest.mark.parametrize("max_ctx", [513, 1025, 4096, 20000])
def test_default_workspace_covers_every_decode_path(capi, H, Hk, D, max_ctx):
    """pa_decode_workspace_bytes(..., 0) is enough for every entry point at its
    default partition size (512 tokens on the CUDA-core kernel, 1024 on the
    tensor-core one): with that many bytes each call passes every host check
    and only then fails for want of a device (PA_ERR_CUDA); the CUDA-core
    path needs all of it (16 bytes fewer is PA_ERR_WORKSPACE)."""
    B = 8
    wsb = capi.pa_decode_workspace_bytes(B, H, D, max_ctx, 0)
    assert wsb > 0
    p, q, ws = C.c_void_p(4096), C.c_void_p(1 << 16), C.c_void_p(1 << 24)
    maxb = (max_ctx + 15) // 16

    def common(n):
        return (C.c_float(0.1), H, Hk, D, 16, B, maxb, max_ctx, 100000, 0, ws, n, None)

    assert capi.pa_decode_ex(p, q, p, p, p, p, *common(wsb)) == -4
    assert capi.pa_decode_fp8(p, q, p, p, p, p, p, p, *common(wsb)) == -4
    assert capi.pa_decode_window(p, q, p, p, p, p, C.c_float(0.1), H, Hk, D, 16, B, maxb, max_ctx, 100000,
                                 max_ctx, 0, ws, wsb, None) == -4
    if D == 128:
        assert capi.pa_decode_tc(p, q, p, p, p, p, *common(wsb)) == -4
    tensor_default = D == 128 and H // Hk == 8
    if not tensor_default:  # pa_decode_ex runs the CUDA-core kernel: 512-token partitions, all bytes used
        assert capi.pa_decode_ex(p, q, p, p, p, p, *common(wsb - 16)) == -3


def test_default_partition_tokens_without_a_device(capi):
    """Without a visible device the wave rule has no slot count: 512 tokens on
    the CUDA-core kernel, 1024 on the tensor-core kernel (groups of 8 at
    head_dim 128, and E4M3 caches at head_dim 128); bad shapes are refused."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is visible: the rule depends on its SM count")
    assert capi.pa_decode_partition_tokens(64, 32, 8, 128, 4096, -1, 2) == 512
    assert capi.pa_decode_partition_tokens(8, 32, 32, 128, 2048, -1, 2) == 512
    assert capi.pa_decode_partition_tokens(100, 64, 8, 128, 4096, -1, 2) == 1024
    assert capi.pa_decode_partition_tokens(64, 32, 8, 128, 4096, -1, 1) == 1024
    assert capi.pa_decode_partition_tokens(64, 32, 8, 64, 4096, -1, 1) == 512
    assert capi.pa_decode_partition_tokens(4, 6, 4, 128, 100, -1, 2) == -1
    assert capi.pa_decode_partition_tokens(4, 4, 4, 96, 100, -1, 2) == -2
    assert capi.pa_decode_partition_tokens(4, 4, 4, 128, 100, -1, 3) == -1


def _plan_items_model(ctx, Hk, part_blocks, max_blocks, max_parts, window):
    """The decode plan restated: every (partition, kv head, sequence) item
    the partition kernels run (a sequence without partitions keeps p = 0),
    longest partition first, (sequence, kv head, partition) order within a
    length."""
    items = []
    for b, c in enumerate(ctx):
        np_, last = 0, 0
        if c > 0:
            nblk = (c + 15) // 16
            bf = (max(0, c - 1 - window) if window >= 0 else 0) // 16
            np_ = (nblk - bf + part_blocks - 1) // part_blocks
            if nblk > max_blocks or np_ > max_parts:
                nblk = min(nblk, max_blocks)
                bf = min(bf, nblk)
                np_ = min((nblk - bf + part_blocks - 1) // part_blocks, max_parts)
                nblk = min(nblk, bf + np_ * part_blocks)
            if np_ > 0:
                last = (nblk - bf) - (np_ - 1) * part_blocks
        if np_ <= 0:
            np_, last = 1, 0
        for kh in range(Hk):
            for p in range(np_):
                items.append((p, kh, b, part_blocks if p + 1 < np_ else last))
    items.sort(key=lambda t: -t[3])   # stable
    return [t[:3] for t in items]


@pytest.mark.parametrize("window", [-1, 300])
def test_decode_plan_matches_model(capi, window):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is visible: the default partition size depends on its SM count")
    import paged_kv_cache_59_gb300 as pk
    rng = np.random.default_rng(5)
    for n_seqs, Hk, H in [(1, 1, 1), (7, 8, 32), (64, 8, 32), (33, 2, 16)]:
        ctx = [int(c) for c in rng.integers(0, 4000, n_seqs)]
        ctx[0] = 0                                       # an empty sequence keeps one item
        max_ctx = max(ctx) + 5
        max_blocks = (max_ctx + 15) // 16
        items = pk.pa_decode_plan(ctx, H, Hk, 128, max_blocks, max_ctx, 1 << 20, window=window)
        pt = pk.pa_decode_partition_tokens(n_seqs, H, Hk, 128, max_ctx, window)   # 512, or 1024 at group 8
        max_parts = (max_ctx + pt - 1) // pt
        if window >= 0:
            max_parts = min(max_parts, ((window + 31) // 16 + pt // 16 - 1) // (pt // 16))
        want = _plan_items_model(ctx, Hk, pt // 16, max_blocks, max_parts, window)
        assert [tuple(int(v) for v in r[:3]) for r in items] == want
        assert (items[:, 3] == 0).all()


def test_decode_plan_errors(capi):
    ctx = (C.c_int32 * 3)(100, 2000, 5)
    buf = (C.c_int32 * 4096)()
    n = capi.pa_decode_plan(ctx, 3, 32, 8, 128, 200, 2000, 4096, -1, 2, 0, None, 0)
    assert n > 0
    assert capi.pa_decode_plan(ctx, 3, 32, 8, 128, 200, 2000, 4096, -1, 2, 0, buf, n - 1) == -8   # capacity
    assert capi.pa_decode_plan(ctx, 3, 32, 8, 128, 200, 2000, 4096, -1, 2, 0, buf, n) == n
    assert capi.pa_decode_plan(ctx, 3, 32, 8, 96, 200, 2000, 4096, -1, 2, 0, buf, n) == -2      # head_dim
    assert capi.pa_decode_plan(ctx, 3, 32, 6, 128, 200, 2000, 4096, -1, 2, 0, buf, n) == -1     # 32 % 6
    assert capi.pa_decode_plan(ctx, 3, 32, 8, 128, 200, 2000, 4096, -1, 3, 0, buf, n) == -1     # elem_bytes
    assert capi.pa_decode_plan(ctx, 3, 32, 8, 128, 200, 2000, 4096, -1, 2, 100, buf, n) == -1   # not a multiple of 64
    assert capi.pa_decode_plan(None, 3, 32, 8, 128, 200, 2000, 4096, -1, 2, 0, buf, n) == -1
