"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a runtime whose HBM is all handed to its KV pool, a decode loop
that must not call cudaMalloc/cudaFree because they can synchronize the
device, a host holding only raw pointers) cannot provide pa_decode's split-K
workspace; this entry point uses a fixed scratch array inside the library
instead. The tests call it through the C ABI and compare it with the
regular pa_decode on two calls in a row (different batches, so a stale
scratch from the first call cannot make the second pass), and check that a
batch too large for the fixed scratch is refused. This file is collected
last so that a failure here stops a -x run only after every other test ran.
"""
import ctypes as C

import numpy as np
import pytest

from tests._gpu import assert_attention_close, bf16_to_f64, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE = -3


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


def _noalloc_via_c_abi(lib, wl, kp, vp):
    torch = torch_cuda()
    q, tabs, ctx = dev(wl.q), dev(wl.dec_tables), dev(wl.dec_ctx)
    out = torch.full_like(q, 0x7FC0)  # NaN-filled: every element must be written
    stream = torch.cuda.current_stream()
    st = lib.pa_decode_noalloc(_vp(out), _vp(q), _vp(kp), _vp(vp), _vp(tabs), _vp(ctx),
                               C.c_float(wl.scale), wl.n_heads, wl.n_kv_heads, wl.head_dim, 16,
                               len(wl.dec_ctx), wl.dec_tables.shape[1], int(wl.dec_ctx.max()),
                               wl.num_blocks, C.c_void_p(stream.cuda_stream))
    assert st == 0, f"pa_decode_noalloc returned {st}"
    torch.cuda.synchronize()
    return host_bits(out)


def test_noalloc_matches_pa_decode_on_two_calls(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as pk
    pk.pa_get_device_error()
    # contexts span 1..9 partitions of 512 tokens, so the split-K scratch is used
    cases = [make_decode_case(601, [3000, 17, 1, 2049, 700, 4096, 512, 513], 32, 8, 128),
             make_decode_case(602, [1500, 4500, 33, 1024, 2], 16, 2, 64)]
    for wl in cases:
        kp, vp = dev(wl.k_pool), dev(wl.v_pool)
        want = _regular(pk, wl, kp, vp)
        got = _noalloc_via_c_abi(capi, wl, kp, vp)
        assert_attention_close(got, bf16_to_f64(want), f"noalloc vs pa_decode ({wl.head_dim})")
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
    assert capi.pa_decode_workspace_bytes(n_seqs, 8, 128, max_ctx, 0) > (32 << 20)
