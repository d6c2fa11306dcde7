"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a runtime whose HBM is all handed to its KV pool, a decode loop
that must not call cudaMalloc/cudaFree because they can synchronize the
device, a host holding only raw pointers) cannot provide pa_decode's split-K
workspace; this entry point uses a fixed scratch array inside the library
instead. The tests call it through the C ABI on two calls in a row (different
batches, so a stale scratch from the first call cannot make the second pass)
and compare every output with the fp64 oracle within the decode tolerance,
and with the regular pa_decode (same kernels, same partitions: the same
bits). The cases reach both partition kernels: the CUDA-core kernel with
512-token partitions and the tensor-core kernel (8 query heads per KV head
at head_dim 128) with 1024-token partitions. Batches too large for the fixed
scratch are refused, at the exact boundary. This file is collected last so
that a failure here stops a -x run only after every other test ran.
"""
import ctypes as C

import numpy as np
import pytest

from oracle.attention import paged_decode
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE = -3
SCRATCH_BYTES = 32 << 20


def _vp(t):
    return C.c_void_p(t.data_ptr())


def _regular(pk, wl, kp, vp):
    torch = torch_cuda()
    q = dev(wl.q)
    out = torch.empty_like(q)
    max_ctx = int(wl.dec_ctx.max())
    ws = pk.decode_workspace(q, max_ctx)
    pk.pa_decode(out, q, kp, vp, dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale, max_ctx, workspace=ws)
    torch.cuda.synchronize()
    return host_bits(out)


def _noalloc_via_c_abi(lib, wl, kp, vp, max_ctx=None):
    torch = torch_cuda()
    q, tabs, ctx = dev(wl.q), dev(wl.dec_tables), dev(wl.dec_ctx)
    out = torch.full_like(q, 0x7FC0)  # NaN-filled: every element must be written
    stream = torch.cuda.current_stream()
    st = lib.pa_decode_noalloc(_vp(out), _vp(q), _vp(kp), _vp(vp), _vp(tabs), _vp(ctx),
                               C.c_float(wl.scale), wl.n_heads, wl.n_kv_heads, wl.head_dim, 16,
                               len(wl.dec_ctx), wl.dec_tables.shape[1],
                               int(max_ctx if max_ctx is not None else wl.dec_ctx.max()),
                               wl.num_blocks, C.c_void_p(stream.cuda_stream))
    assert st == 0, f"pa_decode_noalloc returned {st}"
    torch.cuda.synchronize()
    return host_bits(out)


def test_noalloc_matches_oracle_on_two_calls(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as pk
    pk.pa_get_device_error()
    # contexts span 1..9 partitions of 512 tokens (CUDA-core kernel: groups 4
    # and 8 at head_dim 64) and 1..5 partitions of 1024 tokens (tensor-core
    # kernel: group 8 at head_dim 128), so the split-K scratch is used
    cases = [make_decode_case(601, [3000, 17, 1, 2049, 700, 4096, 512, 513], 32, 8, 128),
             make_decode_case(602, [1500, 4500, 33, 1024, 2], 16, 2, 64),
             make_decode_case(604, [4500, 1025, 1, 3071, 1024, 2048, 9], 64, 8, 128)]
    for wl in cases:
        kp, vp = dev(wl.k_pool), dev(wl.v_pool)
        got = _noalloc_via_c_abi(capi, wl, kp, vp)
        ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
        what = f"noalloc vs oracle (group {wl.group}, head_dim {wl.head_dim})"
        assert_attention_close(got, ref, what)
        want = _regular(pk, wl, kp, vp)
        assert np.array_equal(got, want), f"{what}: differs from pa_decode on the same partitions"
    check_device_error(0)


def test_noalloc_refuses_batches_beyond_its_scratch(capi):
    torch = torch_cuda()
    wl = make_decode_case(603, [40, 9], 8, 8, 128)
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    q, tabs, ctx = dev(wl.q), dev(wl.dec_tables), dev(wl.dec_ctx)
    out = torch.empty_like(q)
    # declared bounds of 2 sequences x 8 heads x 4M tokens: 8192 partitions of
    # (128 + 2) floats per row, ~68 MB of scratch, more than the 32 MiB array
    n_seqs, max_ctx = 2, 1 << 22
    big_tabs = torch.zeros((n_seqs, max_ctx // 16), dtype=torch.int32, device="cuda")
    st = capi.pa_decode_noalloc(_vp(out), _vp(q), _vp(kp), _vp(vp), _vp(big_tabs), _vp(ctx),
                                C.c_float(wl.scale), 8, 8, 128, 16, n_seqs, max_ctx // 16, max_ctx,
                                wl.num_blocks, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == PA_ERR_WORKSPACE
    assert capi.pa_decode_workspace_bytes(n_seqs, 8, 128, max_ctx, 0) > SCRATCH_BYTES


def test_noalloc_scratch_boundary_on_the_tensor_core_path(capi):
    """8 sequences x 64 query heads (group 8, head_dim 128): the largest
    declared context whose workspace fits the 32 MiB scratch runs and matches
    the oracle; one 512-token partition more is refused."""
    torch = torch_cuda()
    n_seqs, H = 8, 64
    fits = 0
    for c in range(512, 1 << 20, 512):
        if capi.pa_decode_workspace_bytes(n_seqs, H, 128, c, 0) > SCRATCH_BYTES:
            break
        fits = c
    assert fits > 0 and capi.pa_decode_workspace_bytes(n_seqs, H, 128, fits + 1, 0) > SCRATCH_BYTES
    wl = make_decode_case(605, [2500, 1, 1100, 64, 777, 2049, 300, 1024], H, 8, 128)
    # tables padded to the declared bound (entries past each context are never read)
    tabs = np.full((n_seqs, (fits + 1 + 15) // 16), -1, dtype=np.int32)
    tabs[:, :wl.dec_tables.shape[1]] = wl.dec_tables
    wl.dec_tables = tabs
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    got = _noalloc_via_c_abi(capi, wl, kp, vp, max_ctx=fits)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(got, ref, "noalloc at the scratch boundary")
    q, t, ctx = dev(wl.q), dev(tabs), dev(wl.dec_ctx)
    out = torch.empty_like(q)
    st = capi.pa_decode_noalloc(_vp(out), _vp(q), _vp(kp), _vp(vp), _vp(t), _vp(ctx), C.c_float(wl.scale),
                                H, 8, 128, 16, n_seqs, tabs.shape[1], fits + 1, wl.num_blocks,
                                C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == PA_ERR_WORKSPACE
    check_device_error(0)
