"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up, reports PA_DEVERR_TIMEOUT through the device error word,
and leaves the CUDA context usable for the next call."""
import ctypes as C

import numpy as np
import pytest

from oracle.attention import paged_decode
from tests._gpu import assert_attention_close, dev, host_bits, torch_cuda
from workloads import make_decode_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(capi):
    torch = torch_cuda()
    import paged_kv_cache_59_gb300 as pk
    pk.pa_get_device_error()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert capi.pa_selftest_wait_timeout(0, stream) == -1          # argument check
    assert capi.pa_selftest_wait_timeout(2000, stream) == 0         # 2 ms limit
    torch.cuda.synchronize()
    assert pk.pa_get_device_error() == 4                            # PA_DEVERR_TIMEOUT
    assert pk.pa_get_device_error() == 0                            # read-and-clear
    # the context is intact: a decode right after gives the oracle's answer
    wl = make_decode_case(901, [33, 700], 8, 2, 128)
    q = dev(wl.q)
    out = torch.empty_like(q)
    pk.pa_decode(out, q, dev(wl.k_pool), dev(wl.v_pool), dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale,
                 700, workspace=pk.decode_workspace(q, 700))
    torch.cuda.synchronize()
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(host_bits(out), ref, "decode after a timeout")
    assert pk.pa_get_device_error() == 0
