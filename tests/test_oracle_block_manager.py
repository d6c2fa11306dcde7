"""Pins for the block-manager reference model (CPU only): the pages' worked
copy-on-write example, their allocation rules and refcount invariants."""
import random

import pytest

from oracle.block_manager import BlockManagerError, BlockManagerModel, OutOfBlocks
from tests.conftest import read_golden


def test_allocates_on_block_boundaries_only():
    """A block is allocated for token 0, 16, 32, ... and not in between."""
    bm = BlockManagerModel(8, 16)
    bm.add_seq(1)
    free0 = bm.num_free()
    for n in range(1, 50):
        bm.append_tokens(1, 1)
        assert free0 - bm.num_free() == (n + 15) // 16
    bm.check_invariants()


def test_slots_follow_table():
    bm = BlockManagerModel(8, 16)
    bm.add_seq(0)
    slots, cow = bm.append_tokens(0, 40)
    assert cow == []
    tab = bm.block_table(0)
    assert slots == [tab[p // 16] * 16 + p % 16 for p in range(40)]


def test_printed_cow_example_refcounts():
    """The three-table figure: b0..b2 shared by A, B, C (refcount 3)."""
    rows = read_golden("cow_sharing.txt")
    seqs = {r[1]: [int(x) for x in r[2:]] for r in rows if r[0] == "seq"}
    refs = {int(r[1]): int(r[2]) for r in rows if r[0] == "ref"}
    prompt = [r for r in rows if r[0] == "prompt"][0]
    assert (int(prompt[1]) + 15) // 16 == int(prompt[2])
    # Build the figure with the manager: A owns a 48-token prompt, B and C fork
    # from it; then each appends private tokens.
    bm = BlockManagerModel(10, 16)
    bm.add_seq(0)
    bm.append_tokens(0, 48)
    bm.fork(0, 1)
    bm.fork(0, 2)
    tails = {0: 32, 1: 32, 2: 16}        # A, B: two more blocks; C: one more
    for s, n in tails.items():
        _, cow = bm.append_tokens(s, n)
        assert cow == []                  # shared blocks are full: no copy
    shared = bm.block_table(0)[:3]
    for s in range(3):
        assert bm.block_table(s)[:3] == shared
    # map the manager's ids onto the figure's ids and compare refcounts
    fig = {name: tab for name, tab in seqs.items()}
    mapping = {}
    for s, name in enumerate(["A", "B", "C"]):
        for mine, theirs in zip(bm.block_table(s), fig[name]):
            assert mapping.setdefault(mine, theirs) == theirs
    for mine, theirs in mapping.items():
        assert bm.refcount(mine) == refs[theirs]
    assert sum(refs.values()) == sum(len(t) for t in fig.values())
    bm.check_invariants()


def test_printed_prefix_sharing_savings():
    row = [r for r in read_golden("cow_sharing.txt") if r[0] == "prefix"][0]
    n_req, pre, tok_b, dup_gib, shared_mib = (int(x) for x in row[1:])
    assert n_req * pre * tok_b / 2 ** 30 == dup_gib
    assert pre * tok_b / 2 ** 20 == shared_mib
    bm = BlockManagerModel(40 + n_req, 16)
    bm.add_seq(0)
    bm.append_tokens(0, pre)
    for r in range(1, n_req):
        bm.fork(0, r)
    assert all(bm.refcount(b) == n_req for b in bm.block_table(0))
    assert 40 + n_req - bm.num_free() == pre // 16      # the pool pays once


def test_write_into_shared_partial_block_copies_first():
    bm = BlockManagerModel(6, 16)
    bm.add_seq(0)
    bm.append_tokens(0, 20)               # block 2 holds 4 tokens
    bm.fork(0, 1)
    last = bm.block_table(0)[1]
    assert bm.refcount(last) == 2
    slots, cow = bm.append_tokens(1, 1)
    assert len(cow) == 1 and cow[0][0] == last
    fresh = cow[0][1]
    assert bm.block_table(1)[1] == fresh and bm.block_table(0)[1] == last
    assert bm.refcount(last) == 1 and bm.refcount(fresh) == 1
    assert slots == [fresh * 16 + 4]
    _, cow2 = bm.append_tokens(0, 1)      # the parent's block is private again
    assert cow2 == []
    bm.check_invariants()


def test_free_only_at_refcount_zero():
    bm = BlockManagerModel(4, 16)
    bm.add_seq(0)
    bm.append_tokens(0, 16)
    b = bm.block_table(0)[0]
    bm.fork(0, 1)
    bm.fork(0, 2)
    bm.free_seq(0)
    assert bm.refcount(b) == 2 and b not in bm.free
    bm.free_seq(1)
    assert bm.refcount(b) == 1 and b not in bm.free
    bm.free_seq(2)
    assert bm.refcount(b) == 0 and b in bm.free
    bm.check_invariants()


def test_out_of_blocks_changes_nothing():
    bm = BlockManagerModel(2, 16)
    bm.add_seq(0)
    bm.append_tokens(0, 20)
    before = (bm.block_table(0), bm.num_free(), bm.seq_len(0))
    with pytest.raises(OutOfBlocks):
        bm.append_tokens(0, 13)           # needs a third block
    assert (bm.block_table(0), bm.num_free(), bm.seq_len(0)) == before
    bm.append_tokens(0, 12)               # exactly fills block 2
    assert bm.num_free() == 0


def test_errors():
    bm = BlockManagerModel(2, 16)
    bm.add_seq(0)
    with pytest.raises(BlockManagerError):
        bm.add_seq(0)
    with pytest.raises(BlockManagerError):
        bm.free_seq(9)
    with pytest.raises(BlockManagerError):
        bm.fork(9, 10)
    with pytest.raises(BlockManagerError):
        bm.append_tokens(5, 1)


def test_random_operation_sequences_keep_invariants():
    rng = random.Random(0)
    for trial in range(30):
        bm = BlockManagerModel(rng.randint(4, 40), 16)
        live = []
        next_id = 0
        for _ in range(200):
            op = rng.random()
            try:
                if op < 0.2 or not live:
                    bm.add_seq(next_id); live.append(next_id); next_id += 1
                elif op < 0.6:
                    bm.append_tokens(rng.choice(live), rng.randint(0, 40))
                elif op < 0.75:
                    bm.fork(rng.choice(live), next_id); live.append(next_id); next_id += 1
                elif op < 0.85:
                    s = rng.choice(live)
                    if bm.block_table(s):
                        bm.make_private(s, rng.randrange(len(bm.block_table(s))))
                else:
                    s = rng.choice(live); bm.free_seq(s); live.remove(s)
            except OutOfBlocks:
                pass
            bm.check_invariants()
        for s in list(live):
            bm.free_seq(s)
        assert bm.num_free() == len(bm.ref)
