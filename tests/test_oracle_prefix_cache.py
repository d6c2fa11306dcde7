"""Pins for the prefix cache of the block-manager model (CPU).

The model's lookup is tied to a brute-force search for the longest cached
prefix of whole blocks (the page's lookup walks prefix lengths from the
longest down and returns the first one it finds); sharing is tied to the
closed forms of the shared-system-prompt example; eviction to a hand-worked
LRU order; everything to the refcount invariants.
"""
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks


def _brute_force_cached_len(registered, tokens, bs=16):
    """Longest n*bs such that tokens[:n*bs] is a registered prefix, trying n
    from the largest possible down (as the page's lookup does)."""
    for n in range(len(tokens) // bs, 0, -1):
        if tuple(tokens[:n * bs]) in registered:
            return n * bs
    return 0


def _serve(m, seq, tokens):
    """Admit a request: reuse the cached prefix, append the rest, cache it."""
    got = m.add_seq_cached(seq, tokens)
    m.append_tokens(seq, len(tokens) - got)
    m.cache_full_blocks(seq, tokens)
    return got


def test_shared_system_prompt_is_computed_once():
    """N requests (the page speaks of 1,000 users; 200 here) with the same
    2,048-token system prompt plus a distinct 37-token query: the first
    computes the prompt's 128 blocks, every later one finds all 2,048 tokens
    cached and allocates only its 3 query blocks."""
    N = 200
    rng = np.random.default_rng(0)
    prompt = [int(t) for t in rng.integers(0, 32000, 2048)]
    m = BlockManagerModel(128 + N * 3, 16)
    cached = []
    for r in range(N):
        query = [int(t) for t in rng.integers(0, 32000, 37)]
        cached.append(_serve(m, r, prompt + query))
    assert cached[0] == 0 and all(c == 2048 for c in cached[1:])
    assert m.num_free() == 0                      # 128 + N * 3 blocks exactly
    prompt_blocks = m.block_table(0)[:128]
    assert all(m.block_table(r)[:128] == prompt_blocks for r in range(N))
    assert all(m.refcount(b) == N + 1 for b in prompt_blocks)      # tables + cache
    # each request's two full query blocks (tokens 2048..2079) are cached under
    # that request's own prefix; its third, partial block is not
    assert m.num_cached() == 128 + N * 2
    m.check_invariants()


def test_lookup_matches_brute_force_longest_prefix():
    rng = random.Random(3)
    base = [rng.randrange(50) for _ in range(200)]
    m = BlockManagerModel(400, 16)
    registered = set()
    seq = 0
    for trial in range(120):
        cut = rng.randrange(0, 200)
        tokens = base[:cut] + [rng.randrange(50) for _ in range(rng.randrange(0, 60))]
        want = _brute_force_cached_len(registered, tokens)
        assert len(m.lookup(tokens)) * 16 == want
        if rng.random() < 0.5 and len(tokens) >= 1:
            got = _serve(m, seq, tokens)
            assert got == want
            for n in range(1, len(tokens) // 16 + 1):
                registered.add(tuple(tokens[:n * 16]))
            m.free_seq(seq)
            seq += 1
        m.check_invariants()


def test_partial_blocks_are_not_cached_and_divergence_shares_earlier_blocks():
    m = BlockManagerModel(32, 16)
    a = list(range(100, 150))                     # 50 tokens: 3 full blocks + 2
    assert _serve(m, 0, a) == 0
    assert m.num_cached() == 3
    b = a[:40] + [999] + a[41:]                   # diverges inside block 2
    assert m.add_seq_cached(1, b) == 32           # blocks 0, 1 only
    assert m.block_table(1) == m.block_table(0)[:2]
    m.check_invariants()


def test_lru_eviction_order_and_pinning():
    """Pool of 6 blocks. Prompts A, B, C of one block each are served and
    freed, so the cache holds them alone, oldest A. A lookup of A refreshes it
    (order B, C, A); with A released again, a need for 4 blocks takes the 3
    free ones and evicts B, the next need evicts C; an entry whose block a
    live table holds is skipped, and goes once that table is freed."""
    bs = 16
    A, B, C = [list(range(k, k + bs)) for k in (0, 100, 200)]
    m = BlockManagerModel(6, bs)
    for i, t in enumerate((A, B, C)):
        _serve(m, i, t)
        m.free_seq(i)
    assert m.num_free() == 3 and m.num_cached() == 3
    assert m.add_seq_cached(10, A) == 16          # refreshes A
    m.free_seq(10)                                # A is cache-only again
    m.add_seq(11)
    m.append_tokens(11, 4 * bs)                   # 3 free + evict B (least recent)
    assert set(m.cache) == {tuple(A), tuple(C)}
    m.append_tokens(11, bs)                       # evicts C
    assert set(m.cache) == {tuple(A)}
    assert m.add_seq_cached(12, A) == 16          # a live table holds A
    with pytest.raises(OutOfBlocks):
        m.append_tokens(11, bs)
    m.free_seq(12)
    m.append_tokens(11, bs)                       # now A goes
    assert m.num_cached() == 0
    m.check_invariants()


def test_appends_are_all_or_nothing_with_eviction():
    m = BlockManagerModel(4, 16)
    _serve(m, 0, list(range(32)))                 # 2 blocks cached, held
    m.free_seq(0)                                 # now evictable
    m.add_seq(1)
    with pytest.raises(OutOfBlocks):
        m.append_tokens(1, 5 * 16)                # needs 5 > 2 free + 2 evictable
    assert m.num_cached() == 2 and m.num_free() == 2   # nothing changed
    m.append_tokens(1, 4 * 16)
    assert m.num_cached() == 0 and m.num_free() == 0
    m.check_invariants()


def test_random_operations_keep_invariants():
    rng = random.Random(17)
    m = BlockManagerModel(40, 16)
    prompts = [[rng.randrange(20) for _ in range(rng.randrange(1, 90))] for _ in range(8)]
    live = {}
    nxt = 0
    for _ in range(600):
        op = rng.random()
        try:
            if op < 0.4:
                t = list(rng.choice(prompts)) + [rng.randrange(20) for _ in range(rng.randrange(0, 20))]
                _serve(m, nxt, t)
                live[nxt] = t
                nxt += 1
            elif op < 0.6 and live:
                s = rng.choice(list(live))
                extra = [rng.randrange(20) for _ in range(rng.randrange(1, 20))]
                m.append_tokens(s, len(extra))
                live[s] = live[s] + extra
                m.cache_full_blocks(s, live[s])
            elif op < 0.7 and live:
                s = rng.choice(list(live))
                m.fork(s, nxt)
                live[nxt] = list(live[s])
                nxt += 1
            elif live:
                s = rng.choice(list(live))
                m.free_seq(s)
                del live[s]
        except OutOfBlocks:
            # a failed admission leaves its (empty or partial) sequence behind: drop it
            for s in [s for s in m.tables if s not in live]:
                m.free_seq(s)
        m.check_invariants()
        cached_blocks = list(m.cache.values())
        assert len(cached_blocks) == len(set(cached_blocks))    # a block is cached at most once
