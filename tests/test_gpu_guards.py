"""Guard bytes around the outputs and the workspaces.

compute-sanitizer is not available, so out-of-bounds writes are looked for
directly: `out` and the workspace are carved out of larger buffers whose
4 KiB head and tail hold a fixed byte pattern, and after the call the pattern
must be intact. The results are also checked against the oracle, so a write
that lands inside the buffer but in the wrong place shows up too.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode, paged_prefill
from oracle.cache_ops import reshape_and_cache as o_rac
from oracle.fp8 import paged_decode_fp8
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case, make_decode_case_fp8, make_prefill_case

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def _guarded(nbytes):
    """A byte buffer with guards on both sides, and its middle nbytes."""
    torch = torch_cuda()
    buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_intact(buf):
    b = buf.cpu().numpy()
    return bool((b[:GUARD] == PATTERN).all() and (b[-GUARD:] == PATTERN).all())


@pytest.mark.parametrize("H,Hk,tc,pt", [(32, 8, False, 64), (32, 8, True, 64), (64, 8, False, 0), (8, 8, False, 128)])
def test_decode_writes_stay_inside(pk, H, Hk, tc, pt):
    torch = torch_cuda()
    ctx = [1, 17, 300, 1000, 2049]
    D = 128
    wl = make_decode_case(61 + H + Hk + pt, ctx, H, Hk, D)
    n = len(ctx)
    out_buf, out_bytes = _guarded(n * H * D * 2)
    out = out_bytes.view(torch.int16).view(n, H, D)
    wsb = pk.pa_decode_workspace_bytes(n, H, D, max(ctx), pt)
    ws_buf, ws = _guarded(wsb)
    pk.pa_decode(out, dev(wl.q), dev(wl.k_pool), dev(wl.v_pool), dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale,
                 max(ctx), workspace=ws, partition_tokens=pt, tensor_cores=tc)
    torch.cuda.synchronize()
    assert _guards_intact(out_buf), "decode wrote outside out"
    assert _guards_intact(ws_buf), "decode wrote outside the workspace"
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(host_bits(out), ref, f"guarded decode H={H} Hk={Hk} tc={tc}")
    check_device_error(0)


@pytest.mark.parametrize("pt", [0, 64])
def test_fp8_decode_writes_stay_inside(pk, pt):
    """The E4M3 tensor-core kernel (V widened in registers, outputs in a
    permuted dims order put back by its epilogue)."""
    torch = torch_cuda()
    ctx = [1, 17, 300, 1000, 2049]
    H, Hk, D = 32, 8, 128
    wl = make_decode_case_fp8(63 + pt, ctx, H, Hk, D, n_new=0)
    n = len(ctx)
    out_buf, out_bytes = _guarded(n * H * D * 2)
    out = out_bytes.view(torch.int16).view(n, H, D)
    wsb = pk.pa_decode_workspace_bytes(n, H, D, max(ctx), pt)
    ws_buf, ws = _guarded(wsb)
    pk.pa_decode_fp8(out, dev(wl.q), dev(wl.k_pool), dev(wl.v_pool), dev(wl.meta["k_scale"]),
                     dev(wl.meta["v_scale"]), dev(wl.dec_tables), dev(wl.dec_ctx), wl.scale, max(ctx),
                     workspace=ws, partition_tokens=pt)
    torch.cuda.synchronize()
    assert _guards_intact(out_buf), "fp8 decode wrote outside out"
    assert _guards_intact(ws_buf), "fp8 decode wrote outside the workspace"
    ref = paged_decode_fp8(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale, wl.meta["k_scale"],
                           wl.meta["v_scale"])
    assert_attention_close(host_bits(out), ref, f"guarded fp8 decode pt={pt}")
    check_device_error(0)


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("splits", [None, 0, 3])
def test_prefill_writes_stay_inside(pk, splits, head_dim):
    torch = torch_cuda()
    wl = make_prefill_case(62 + head_dim, [300, 129, 40], [37, 129, 40], [], 32, 8, head_dim)
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    q = dev(wl.q_pf)
    rows, H, D = q.shape
    out_buf, out_bytes = _guarded(rows * H * D * 2)
    out = out_bytes.view(torch.int16).view(rows, H, D)
    max_chunk = int(np.max(np.diff(wl.q_start_loc)))
    args = (out, q, kp, vp, dev(wl.pf_tables), dev(wl.pf_ctx), dev(wl.q_start_loc), wl.scale, max_chunk)
    ws_buf = None
    if splits is None:
        pk.pa_prefill_paged(*args)
    else:
        wsb = pk.pa_prefill_workspace_bytes(len(wl.pf_ctx), H, wl.n_kv_heads, max_chunk, splits)
        ws_buf, ws = _guarded(wsb)
        pk.pa_prefill_paged_ex(*args, splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert _guards_intact(out_buf), "prefill wrote outside out"
    if ws_buf is not None:
        assert _guards_intact(ws_buf), "prefill wrote outside the workspace"
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert_attention_close(host_bits(out), ref, f"guarded prefill splits={splits} head_dim={head_dim}")
    check_device_error(0)
