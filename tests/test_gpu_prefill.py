"""GPU parity for the tcgen05 chunked causal prefill against the fp64 oracle.

Tolerance (per element): |gpu - ref| <= 2e-3 + 1e-2 * |ref|. Cases cover a
whole prompt as one chunk, chunks at an offset with ragged lengths and
partial last blocks (NaN-poisoned slots past the context), several key
tiles, every group size, both head dims (64 and 128), padding rows of a
partial query tile, and sampled rows of the full mixed workload (4 chunks of
512 at 32K context).
"""
import numpy as np
import pytest

from oracle.attention import paged_prefill
from oracle.cache_ops import reshape_and_cache as o_rac
from tests._gpu import assert_attention_close, check_device_error, dev, host_bits, torch_cuda
from workloads import make_prefill_case, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk(capi):
    torch_cuda()
    import paged_kv_cache_59_gb300 as m
    m.pa_get_device_error()
    return m


def _run(pk, wl, splits=None):
    """splits None: pa_prefill_paged (no split); else pa_prefill_paged_ex with that count."""
    torch = torch_cuda()
    kp, vp = dev(wl.k_pool), dev(wl.v_pool)
    pk.pa_reshape_and_cache(dev(wl.new_k), dev(wl.new_v), kp, vp, dev(wl.slot_mapping))
    q = dev(wl.q_pf)
    out = torch.full_like(q, 0x7FC0)
    max_chunk = int(np.max(np.diff(wl.q_start_loc)))
    args = (out, q, kp, vp, dev(wl.pf_tables), dev(wl.pf_ctx), dev(wl.q_start_loc), wl.scale, max_chunk)
    if splits is None:
        pk.pa_prefill_paged(*args)
    else:
        ws = pk.prefill_workspace(q, len(wl.pf_ctx), wl.n_kv_heads, max_chunk, splits)
        ws_poison = ws.fill_(0xFF) if ws is not None else None  # no piece may read what it did not write
        pk.pa_prefill_paged_ex(*args, splits=splits, workspace=ws_poison)
    torch.cuda.synchronize()
    return host_bits(out)


@pytest.mark.parametrize("case", [
    dict(ctx=[40], lens=[40], H=4, Hk=4),                 # G=1, whole prompt, one key tile
    dict(ctx=[300, 129], lens=[37, 129], H=32, Hk=8),     # G=4, offsets, partial blocks
    dict(ctx=[520, 77], lens=[200, 5], H=16, Hk=8),       # G=2, several query tiles
    dict(ctx=[700], lens=[33], H=64, Hk=8),               # G=8, 6 key tiles
    dict(ctx=[256, 255, 17], lens=[256, 1, 17], H=32, Hk=8),  # exact tiles, single-row chunk
])
@pytest.mark.parametrize("head_dim", [128, 64])
def test_prefill_matches_oracle(pk, case, head_dim):
    wl = make_prefill_case(700 + sum(case["ctx"]) + head_dim, case["ctx"], case["lens"], [], case["H"], case["Hk"],
                           head_dim)
    got = _run(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    stats = assert_attention_close(got, ref, f"prefill head_dim {head_dim} {case}")
    check_device_error(0)
    print(case, stats)


@pytest.mark.parametrize("head_dim", [128, 64])
def test_prefill_hot_logits(pk, head_dim):
    """q x 16: row maxima grow tile after tile, exercising the O rescale path."""
    wl = make_prefill_case(731 + head_dim, [600], [64], [], 32, 8, head_dim)
    qf = (wl.q_pf.astype(np.uint32) << 16).view(np.float32) * 16.0
    wl.q_pf = ((qf.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    got = _run(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert_attention_close(got, ref, f"prefill hot, head_dim {head_dim}")
    check_device_error(0)


def _group_rows(wl, ek, ev, s, kh, tokens):
    """Oracle outputs of every query head of KV head kh's group for chunk
    tokens `tokens` of sequence s: [len(tokens)][G][D]. The oracle gets one KV
    head's pools and its group's query heads (the head map h // G is then
    the identity onto that one KV head)."""
    G = wl.n_heads // wl.n_kv_heads
    r0 = int(wl.q_start_loc[s])
    rows = [(r0 + t, g) for t in tokens for g in range(G)]
    ref = paged_prefill(wl.q_pf[:, kh * G:(kh + 1) * G], ek[:, kh:kh + 1], ev[:, kh:kh + 1], wl.pf_tables,
                        wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    return np.stack([ref[r0 + t] for t in tokens])


def _check_group(got, wl, ek, ev, s, kh, tokens, what):
    G = wl.n_heads // wl.n_kv_heads
    r0 = int(wl.q_start_loc[s])
    ref = _group_rows(wl, ek, ev, s, kh, tokens)
    sel = got[[r0 + t for t in tokens]][:, kh * G:(kh + 1) * G]
    assert_attention_close(sel, ref, what)


def _query_tile(G, which):
    """Chunk tokens of one complete 128-row query tile (128 / G tokens x G heads)."""
    qt = 128 // G
    return list(range(which * qt, (which + 1) * qt))


def test_prefill_mixed_workload_sampled_rows(pk):
    wl = make_workload("mixed")
    got = _run(pk, wl)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rng = np.random.default_rng(4)
    n_rows = int(wl.q_start_loc[-1])
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, n_rows, 24), rng.integers(0, 32, 24))]
    rows += [(0, 0), (511, 31), (512, 5), (n_rows - 1, 7)]   # chunk edges
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    for r, h in rows:
        assert_attention_close(got[r, h], ref[r, h], f"mixed prefill row {(r, h)}")
    # complete query tiles: the chunk start of the first sequence, the chunk end of the last
    G = wl.n_heads // wl.n_kv_heads
    L = int(wl.q_start_loc[1] - wl.q_start_loc[0])
    _check_group(got, wl, ek, ev, 0, 1, _query_tile(G, 0), "mixed prefill: chunk-start tile")
    _check_group(got, wl, ek, ev, len(wl.pf_ctx) - 1, 6, _query_tile(G, L * G // 128 - 1),
                 "mixed prefill: chunk-end tile")
    check_device_error(0)


@pytest.mark.parametrize("splits", [0, 2, 3, 5, 8, 13])   # the merge combines up to 8 pieces in one round, more in batches
@pytest.mark.parametrize("case", [
    dict(ctx=[300, 129], lens=[37, 129], H=32, Hk=8),     # G=4, offsets, partial blocks (few key tiles)
    dict(ctx=[700], lens=[33], H=64, Hk=8),               # G=8, 6 key tiles
    dict(ctx=[1500, 40], lens=[300, 40], H=16, Hk=8),     # G=2, pieces of a long range and empty pieces
])
def test_prefill_split_pieces_match_oracle(pk, case, splits):
    """Key ranges split into pieces (including more pieces than key tiles, so
    some are empty) and merged give the unsplit result's accuracy."""
    wl = make_prefill_case(800 + sum(case["ctx"]) + splits, case["ctx"], case["lens"], [], case["H"], case["Hk"],
                           128)
    got = _run(pk, wl, splits)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert_attention_close(got, ref, f"prefill split={splits} {case}")
    check_device_error(0)


@pytest.mark.parametrize("splits", [0, 3])
def test_prefill_split_pieces_head_dim_64(pk, splits):
    """The merge at head_dim 64 (two dims per lane): pieces of long key
    ranges, empty pieces, every group size in one batch of sequences."""
    for G, (ctx, lens) in {1: ([900, 33], [130, 33]), 8: ([1500, 40], [300, 40])}.items():
        wl = make_prefill_case(860 + G + splits, ctx, lens, [], 8 * G, 8, 64)
        got = _run(pk, wl, splits)
        ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
        ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
        assert_attention_close(got, ref, f"prefill head_dim 64 group {G} split={splits}")
    check_device_error(0)


def _balanced_cut(n_pairs, n_cta):
    """The balanced work list's rule for where whole pairs end: with P
    non-empty pairs and C CTAs, the last R = P mod C pairs are cut into S key
    ranges, S in 1..8 with R*S <= 4C minimising ceil(R*S/C)/S + 0.03 S (no
    cut when S = 1). Returns (first cut pair, S)."""
    R = n_pairs % n_cta
    best, S = 2.0, 1
    for c in range(1, 9):
        if R * c > 4 * n_cta:
            break
        cost = -(-R * c // n_cta) / c + 0.03 * c
        if cost < best:
            best, S = cost, c
    return (n_pairs - R if S > 1 else n_pairs), S


def test_prefill_mixed_workload_auto_split_tiles(pk):
    """Balanced mode on the full mixed batch: every query head of a complete
    query tile at the chunk start and at the chunk end of every long
    sequence, both query tiles of the last pair that runs whole and of the
    first pair cut into key-range pieces, and random rows."""
    torch = torch_cuda()
    wl = make_workload("mixed")
    got = _run(pk, wl, 0)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    G = wl.n_heads // wl.n_kv_heads
    Hk = wl.n_kv_heads
    L = int(wl.q_start_loc[1] - wl.q_start_loc[0])
    assert all(int(wl.q_start_loc[i + 1] - wl.q_start_loc[i]) == L for i in range(len(wl.pf_ctx)))
    for s in range(len(wl.pf_ctx)):
        _check_group(got, wl, ek, ev, s, (2 * s) % Hk, _query_tile(G, 0), f"seq {s}: chunk-start tile")
        _check_group(got, wl, ek, ev, s, (2 * s + 1) % Hk, _query_tile(G, L * G // 128 - 1),
                     f"seq {s}: chunk-end tile")
    # pair items in work-list order: (sequence * Hk + kv head) * pairs_per_seq + pair
    n_qp = L * G // 256
    n_items = len(wl.pf_ctx) * Hk * n_qp
    first_cut, S = _balanced_cut(n_items, torch.cuda.get_device_properties(0).multi_processor_count)
    assert S > 1 and 0 < first_cut < n_items, "the mixed batch's last partial wave is expected to be cut"
    for it, what in ((first_cut - 1, "last whole pair"), (first_cut, f"first pair cut into {S} pieces")):
        s, kh, qp = it // (Hk * n_qp), (it // n_qp) % Hk, it % n_qp
        toks = list(range(qp * 256 // G, (qp + 1) * 256 // G))
        _check_group(got, wl, ek, ev, s, kh, toks, f"{what} (seq {s}, kv head {kh}, pair {qp})")
    rng = np.random.default_rng(6)
    n_rows = int(wl.q_start_loc[-1])
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, n_rows, 24), rng.integers(0, 32, 24))]
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    for r, h in rows:
        assert_attention_close(got[r, h], ref[r, h], f"mixed split prefill row {(r, h)}")
    check_device_error(0)


@pytest.mark.parametrize("seed,n_seqs,ctx_hi,len_hi", [(21, 24, 600, 150), (22, 7, 4000, 300)])
def test_prefill_balanced_shares_cross_pairs(pk, seed, n_seqs, ctx_hi, len_hi):
    """Balanced mode (splits 0) with more key tiles than CTAs: a CTA's share
    starts inside one pair, may hold whole pairs, and ends inside another, so
    both partial slots, direct outputs and multi-piece merges occur; uneven
    sequences leave pairs past the shorter chunks empty."""
    rng = np.random.default_rng(seed)
    ctx = [int(c) for c in rng.integers(50, ctx_hi, n_seqs)]
    lens = [int(min(c, n)) for c, n in zip(ctx, rng.integers(1, len_hi, n_seqs))]
    wl = make_prefill_case(seed, ctx, lens, [], 16, 8, 128)
    got = _run(pk, wl, 0)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert_attention_close(got, ref, f"prefill balanced seed={seed}")
    check_device_error(0)


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_chunk_not_in_cache_is_flagged_and_spares_others(pk, splits):
    """A sequence whose context is shorter than its chunk sets PA_DEVERR_CONTEXT,
    writes nothing, and leaves the other sequence's rows exact (per-pair and
    balanced scheduling)."""
    wl = make_prefill_case(941, [300, 40], [37, 20], [], 32, 8, 128)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rows = [(r, h) for r in range(37) for h in range(32)]
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    wl.pf_ctx = wl.pf_ctx.copy()
    wl.pf_ctx[1] = 10                                   # 20 chunk rows, 10 cached tokens
    got = _run(pk, wl, splits)
    for r, h in rows:
        assert_attention_close(got[r, h], ref[r, h], f"row {(r, h)}")
    assert (got[37:] == 0x7FC0).all()                   # untouched (the pre-filled NaN pattern)
    check_device_error(16)                              # PA_DEVERR_CONTEXT


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_bad_block_id_is_flagged_not_faulted(pk, splits):
    """A block-table entry outside the pool sets PA_DEVERR_BLOCK_ID; that block
    loads as zeros and the other sequence's rows stay exact."""
    wl = make_prefill_case(942, [300, 500], [37, 64], [], 32, 8, 128)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    rows = [(r, h) for r in range(37) for h in range(32)]
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    wl.pf_tables = wl.pf_tables.copy()
    wl.pf_tables[1, 3] = wl.num_blocks + 5             # sequence 1, tokens 48..63
    got = _run(pk, wl, splits)
    for r, h in rows:
        assert_attention_close(got[r, h], ref[r, h], f"row {(r, h)}")
    check_device_error(1)                               # PA_DEVERR_BLOCK_ID


def _scale_bf16(bits, factor):
    """bf16 bits times a power of two (exact; NaN stays NaN)."""
    f = (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_small_v(pk, splits):
    """P.V stages V as fp16 values of v * 2^-8: V of magnitude ~2^-12 (subnormal
    after the scaling) still matches the oracle within the tolerance."""
    wl = make_prefill_case(951, [300, 129], [37, 129], [], 32, 8, 128)
    wl.v_pool = _scale_bf16(wl.v_pool, 2.0 ** -12)
    wl.new_v = _scale_bf16(wl.new_v, 2.0 ** -12)
    got = _run(pk, wl, splits)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert_attention_close(got, ref, "V x 2^-12")
    check_device_error(0)


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_large_v_scales_exactly(pk, splits):
    """Attention is linear in V. P.V stages V as fp16 values of v * 2^-8, which
    holds every bf16 significand exactly while v * 2^-8 is a normal fp16 value
    (2^-14 .. 65504). Here the nonzero |v| span 2^-20.3 .. 5, so V x 2^15 and
    V x 2^21 (values up to ~2^23, far beyond the plain fp16 range) both stage
    exactly, and the outputs differ by exactly 2^6: the bf16 output bits
    differ by 6 in the exponent field only."""
    wl = make_prefill_case(953, [300, 129], [37, 129], [], 32, 8, 128)
    mags = []
    for a in (wl.v_pool, wl.new_v):
        f = np.abs((a.astype(np.uint32) << 16).view(np.float32))
        mags.append(f[np.isfinite(f) & (f > 0)])
    mags = np.concatenate(mags)
    assert mags.min() * 2.0 ** (15 - 8) >= 2.0 ** -14 and mags.max() * 2.0 ** (21 - 8) <= 65504
    v_pool, new_v = wl.v_pool, wl.new_v
    outs = []
    for c in (15, 21):
        wl.v_pool, wl.new_v = _scale_bf16(v_pool, 2.0 ** c), _scale_bf16(new_v, 2.0 ** c)
        outs.append(_run(pk, wl, splits))
        check_device_error(0)
    assert np.array_equal(outs[1], _scale_bf16(outs[0], 2.0 ** 6))


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_v_beyond_fp16_staging_is_flagged(pk, splits):
    """One V element of 2^25 (> 65504 * 2^8) in a key tile the chunk reads:
    the affected outputs are not finite and PA_DEVERR_RANGE is set."""
    wl = make_prefill_case(952, [300], [37], [], 32, 8, 128)
    wl.new_v = wl.new_v.copy()
    wl.new_v[0, 0, 5] = 0x4C00                          # bf16 2^25 at the chunk's first token
    got = _run(pk, wl, splits)
    assert not np.isfinite((got.astype(np.uint32) << 16).view(np.float32)).all()
    check_device_error(64)                              # PA_DEVERR_RANGE


def _bf16(x):
    f = np.asarray(x, np.float32)
    return ((f.view(np.uint32) + 0x7FFF + ((f.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("splits", [None, 0])
def test_prefill_row_maximum_jump_keeps_earlier_keys(pk, splits):
    """One row whose scores jump twice inside one key tile: a key 15 binades
    (log2 units after the scale) above the reference of the first tile, then
    one 25.5 binades above it. The second jump rescales the tile's earlier P
    by about 2^-25, a factor below fp16's range although the rescaled P
    (about 2^-10) is not: the key 15 binades up keeps its weight of about
    2^-10.5, which carries the whole output (its V is 8, every other V is 0)."""
    torch = torch_cuda()
    H = Hk = 4
    D, ctx = 128, 300
    wl = make_prefill_case(960, [ctx], [1], [], H, Hk, D)
    sc = wl.scale / np.log(2.0)                      # scores -> log2 units
    base = 20.0 / sc                                 # first tile's maximum at 20 binades
    x = np.full(ctx, -200.0)                         # every other key: far below
    x[5], x[130], x[230] = base, base + 15.0 / sc, base + 25.5 / sc
    kpos = np.zeros((ctx, Hk, D), np.float32)
    kpos[:, :, 0] = x[:, None]
    vpos = np.zeros((ctx, Hk, D), np.float32)
    vpos[130] = 8.0
    K, V = _bf16(kpos), _bf16(vpos)
    tab = wl.pf_tables[0]
    for t in range(ctx - 1):                         # the cached tokens; the last one is this step's
        wl.k_pool[tab[t // 16], :, t % 16] = K[t]
        wl.v_pool[tab[t // 16], :, t % 16] = V[t]
    wl.new_k = K[ctx - 1:ctx].copy()
    wl.new_v = V[ctx - 1:ctx].copy()
    q = np.zeros((1, H, D), np.float32)
    q[:, :, 0] = 1.0
    wl.q_pf = _bf16(q)
    got = _run(pk, wl, splits)
    ek, ev = o_rac(wl.new_k, wl.new_v, wl.k_pool, wl.v_pool, wl.slot_mapping)
    ref = paged_prefill(wl.q_pf, ek, ev, wl.pf_tables, wl.pf_ctx, wl.q_start_loc, wl.scale)
    assert ref[0, 0, 0] > 3e-3                       # the moderate key's share is not negligible
    assert_attention_close(got, ref, "row maximum jump")
    check_device_error(0)
