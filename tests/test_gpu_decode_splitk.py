"""Split-K workspace of pa_decode.

The workspace needs no initialisation: every partial that the merge reads is
written by the same call. These tests check that through the C ABI on both
partition kernels: outputs against the oracle from poisoned workspaces,
repeated and graph-replayed calls bit-identical to the first, and contexts of
several hundred partitions.

Tolerance (per element): |gpu - ref| <= 2e-3 + 1e-2 * |ref|.
"""
import numpy as np
import pytest

from oracle.attention import paged_decode
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_decode_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def _case(seed, ctx, H=32, Hk=8, D=128):
    wl = make_decode_case(seed, ctx, H, Hk, D)
    ref = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    d = dict(q=dev(wl.q), kp=dev(wl.k_pool), vp=dev(wl.v_pool), tab=dev(wl.dec_tables),
             ctx=dev(wl.dec_ctx))
    return wl, ref, d


def _run(pk, d, wl, ws, pt, tc=False):
    torch = torch_cuda()
    out = torch.empty_like(d["q"])
    pk.pa_decode(out, d["q"], d["kp"], d["vp"], d["tab"], d["ctx"], wl.scale, int(wl.dec_ctx.max()),
                 workspace=ws, partition_tokens=pt, tensor_cores=tc)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("fill", ["zero", "ones", "stale", "nan"])
def test_poisoned_workspace(pk, tc, fill):
    torch = torch_cuda()
    ctx = [1, 17, 600, 1500, 2049, 4000]
    wl, ref, d = _case(31, ctx)
    pt = 256
    n, H, D = wl.q.shape
    nbytes = pk.pa_decode_workspace_bytes(n, H, D, max(ctx), pt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if fill == "zero":
        ws.zero_()
    elif fill == "ones":
        ws.fill_(0xFF)
    elif fill == "nan":
        ws.view(torch.float32).fill_(float("nan"))
    else:  # another call's partials: a larger max and sum than any of this call's
        ws.view(torch.float32).fill_(1e30)
    out = _run(pk, d, wl, ws, pt, tc)
    assert_attention_close(host_bits(out), ref, f"fill={fill} tc={tc}")
    check_device_error(0)


@pytest.mark.parametrize("tc", [False, True])
def test_repeated_calls_bit_identical(pk, tc):
    torch = torch_cuda()
    ctx = [4096, 333, 2048, 1025]
    wl, ref, d = _case(32, ctx)
    n, H, D = wl.q.shape
    ws = torch.empty(pk.pa_decode_workspace_bytes(n, H, D, max(ctx), 128), dtype=torch.uint8, device="cuda")
    first = host_bits(_run(pk, d, wl, ws, 128, tc))
    assert_attention_close(first, ref, "first call")
    for _ in range(4):
        assert np.array_equal(host_bits(_run(pk, d, wl, ws, 128, tc)), first)
    check_device_error(0)


def test_graph_replay(pk):
    """A captured call replays bit-identically to the eager call, and picks up
    new query values written into its input between replays."""
    torch = torch_cuda()
    ctx = [3000, 700, 4096]
    wl, ref, d = _case(33, ctx)
    n, H, D = wl.q.shape
    ws = torch.empty(pk.pa_decode_workspace_bytes(n, H, D, max(ctx), 0), dtype=torch.uint8, device="cuda")
    eager = host_bits(_run(pk, d, wl, ws, 0))
    assert_attention_close(eager, ref, "eager")
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm the binding on the side stream before capture
        pk.pa_decode(out, d["q"], d["kp"], d["vp"], d["tab"], d["ctx"], wl.scale, max(ctx), workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pk.pa_decode(out, d["q"], d["kp"], d["vp"], d["tab"], d["ctx"], wl.scale, max(ctx), workspace=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), eager)
    # new query values through the same graph
    q2 = make_decode_case(34, ctx, H, wl.n_kv_heads, D).q
    d["q"].copy_(dev(q2))
    g.replay()
    torch.cuda.synchronize()
    ref2 = paged_decode(q2, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    assert_attention_close(host_bits(out), ref2, "replay with new q")
    check_device_error(0)


@pytest.mark.parametrize("tc", [False, True])
def test_hundreds_of_partitions(pk, tc):
    """64-token partitions over 20,000 tokens: 313 partials per row, more than
    the merging warp's 32 lanes and 8-wide slice loads cover in one pass."""
    ctx = [20000, 19999, 64, 65]
    wl, ref, d = _case(35, ctx, H=16, Hk=4)
    torch = torch_cuda()
    n, H, D = wl.q.shape
    ws = torch.empty(pk.pa_decode_workspace_bytes(n, H, D, max(ctx), 64), dtype=torch.uint8, device="cuda")
    out = _run(pk, d, wl, ws, 64, tc)
    assert_attention_close(host_bits(out), ref, f"313 partitions tc={tc}")
    check_device_error(0)


def _default_rule(n_seqs, n_kv_heads, span, sms, slots):
    """The CUDA-core kernel's default partition size, restated: one partition
    per sequence when one CTA per (sequence, KV head) covers every SM in a
    single wave and a context fits 2048 tokens; otherwise the multiple of 64
    in [512, 1024] whose grid fills its last wave of CTA slots best."""
    groups = n_seqs * n_kv_heads
    if sms <= groups <= slots and 512 < span <= 2048:
        return -(-span // 64) * 64
    if span <= 512:
        return 512
    best, best_fill = 512, -1.0
    for pt in range(512, 1025, 64):
        waves = groups * -(-span // pt) / slots
        fill = waves / np.ceil(waves)
        if fill > best_fill + 1e-9:
            best, best_fill = pt, fill
    return best


@pytest.mark.parametrize("shape", [
    (8, 32, 32, 128, 2048),    # 7B MHA batch: 256 groups in one wave -> one partition of 2048
    (8, 32, 32, 128, 1500),    # the same at a shorter bound -> 1536
    (64, 32, 8, 128, 4096),    # 8B GQA batch: 512 groups, more than one wave
    (4, 32, 32, 128, 2048),    # 128 groups, fewer than the SMs
    (32, 32, 8, 128, 4096),    # one partition would exceed 2048 tokens
])
def test_default_partition_tokens_follow_the_rule(pk, capi, shape):
    torch = torch_cuda()
    n_seqs, H, Hk, D, ctx = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want = _default_rule(n_seqs, Hk, ctx, sms, 3 * sms)   # 3 CTAs per SM for groups up to 4
    assert pk.pa_decode_partition_tokens(n_seqs, H, Hk, D, ctx) == want


def test_single_partition_default_matches_oracle(pk):
    """Uneven contexts up to 2048 tokens over 160 (sequence, KV head) groups
    of MHA: the default takes one partition per sequence, no merge."""
    torch = torch_cuda()
    rng = np.random.default_rng(77)
    ctx = [2048, 1, 17, 1500] + [int(c) for c in rng.integers(300, 2049, 16)]
    wl, ref, d = _case(711, ctx, H=8, Hk=8, D=128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if not sms <= len(ctx) * 8 <= 3 * sms:
        pytest.skip("the one-partition rule does not apply on this device")
    assert pk.pa_decode_partition_tokens(len(ctx), 8, 8, 128, 2048) == 2048
    assert pk.decode_workspace(d["q"], 2048) is not None       # sized for 512, the bound of every default
    out = torch.full_like(d["q"], 0x7FC0)
    pk.pa_decode(out, d["q"], d["kp"], d["vp"], d["tab"], d["ctx"], wl.scale, 2048)
    torch.cuda.synchronize()
    assert_attention_close(host_bits(out), ref, "one partition per sequence (default)")
    check_device_error(0)
