"""Reference model of the host block manager (free list, refcounts, fork, CoW).

Sources:
* "PagedAttention vs Traditional KV Cache", Section 4 "PagedAttention: How It
  Works": a free list of block ids (allocation pops from it and fails when it
  is empty - the caller then preempts), a per-sequence block table, and
  appending a token allocates a new block only when the last one is full.
* "Inference serving: the KV-cache machine", section "Paged KV: virtual memory
  for tokens" and Lab B's BlockPool: blocks carry a reference count; a block
  returns to the pool only when its count reaches zero; fork makes the child
  table alias the parent's blocks (incref each), and the first divergent token
  gets a private block.
* "Modern AI Infrastructure and Agentic System Design", 9.1, copy-on-write
  figure: three tables share b0..b2 (refcount 3); a write to a shared block
  first copies it into a fresh block.

Readings taken where the pages are silent or disagree:
* The first page's free_sequence returns every block to the free list, which
  would free blocks still shared by a sibling; the refcounted release of the
  other two pages is followed instead.
* refcount = number of block tables that reference the block.
* Appending into a partially filled last block whose refcount > 1 copies it
  first (copy pair emitted, src decref'd, table repointed). If the shared last
  block is full, the new token simply starts a new private block.
* ``make_private`` forces the copy of any shared block of a sequence (used to
  model a divergent overwrite of an already full block).
* An append of n tokens is all-or-nothing: if the free list cannot supply
  every block it needs, nothing changes and OutOfBlocks is raised.
* Allocation order (LIFO pop) is not part of any result the tests compare.
* Sliding window ("KV Cache Explained Like You're an LLM Engineer", section
  "Sliding Window Attention": attention reaches back W tokens, so the cache
  it needs stays O(W)): ``release_before(seq, first)`` drops every block that
  lies wholly before position ``first`` - its table entry becomes the hole -1
  and its refcount drops (the block returns to the free list at zero).
  Positions keep their logical block index, so later appends are unaffected;
  fork, free and the invariants skip holes.
* Prefix caching ("Modular LLM Inference Engine from Scratch", section
  "Prefix caching - skip recomputing the same prompt": a hash-based LRU cache
  whose lookup returns the longest cached prefix made of whole blocks and
  refreshes it; "Inference serving: the KV-cache machine" and "KV Cache
  Explained Like You're an LLM Engineer", section "Prefix Caching": a shared
  prompt's KV is computed once and shared). Reading taken:
  - a cache entry is one full block, keyed by the exact token prefix that
    ends with it (all tokens from position 0 through the block's last), so a
    block is shared only when everything before it matches too;
  - ``cache_full_blocks(seq, tokens)`` registers the sequence's full blocks
    (those whose 16 tokens are all in the sequence); each new entry holds one
    reference to its block and goes to the most-recently-used end; entries
    already present are left where they are;
  - ``add_seq_cached(seq, tokens)`` starts a sequence on the longest run of
    leading blocks whose prefixes are all cached (the longest cached prefix
    of whole blocks), increfs them, sets its length to that many tokens and
    moves those entries to the most-recently-used end, first block first;
  - when an allocation finds the free list empty, entries are evicted from
    the least-recently-used end, skipping entries whose block a table still
    references, until a block is free; an append or a copy succeeds iff the
    free list plus the evictable entries cover it (all-or-nothing);
  - refcount = table references + cache entries.
* Preemption by swapping ("Modern AI Infrastructure and Agentic System
  Design", 9.1, part "Batching and the scheduler": a preempted sequence is
  recomputed later or swapped to host memory; "Inference serving: the
  KV-cache machine", section "Paged KV: virtual memory for tokens": a block
  table makes state movable - swap out the private blocks, reload them later
  anywhere; its Lab B simulator preempts and swaps under this policy).
  Reading taken: ``swap_out(seq)`` releases the sequence's private tail, the
  longest run of trailing blocks that only its table holds (refcount 1), and
  returns them in logical order (the caller copies their contents to host
  memory before anything reuses them); the table keeps the shared head and
  the sequence keeps its length. ``swap_in(seq)`` allocates that many fresh
  blocks (all-or-nothing), appends them to the table and returns them (the
  caller copies the contents back in). A swapped sequence cannot append,
  fork, copy or release until it is swapped in.
"""
from __future__ import annotations

from collections import OrderedDict
from typing import Dict, List, Sequence, Tuple


class OutOfBlocks(Exception):
    pass


class BlockManagerError(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int = 16):
        if num_blocks < 0 or block_size <= 0:
            raise BlockManagerError("bad sizes")
        self.block_size = block_size
        self.free: List[int] = list(range(num_blocks))
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        # prefix cache: exact token prefix (tuple) -> block id, oldest first
        self.cache: "OrderedDict[tuple, int]" = OrderedDict()
        self.swapped: Dict[int, int] = {}   # seq -> blocks held in host memory

    # -- allocation primitives ---------------------------------------------
    def _evictable(self) -> int:
        return sum(1 for b in self.cache.values() if self.ref[b] == 1)

    def available(self) -> int:
        """Blocks an allocation can obtain: free ones plus evictable cache entries."""
        return len(self.free) + self._evictable()

    def _evict_one(self) -> None:
        for key, b in self.cache.items():          # least recently used first
            if self.ref[b] == 1:
                del self.cache[key]
                self._put(b)
                return
        raise OutOfBlocks()

    def _alloc(self) -> int:
        if not self.free:
            self._evict_one()
        b = self.free.pop()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _put(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise BlockManagerError("refcount underflow")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequence operations -----------------------------------------------
    def add_seq(self, seq_id: int) -> None:
        if seq_id in self.tables:
            raise BlockManagerError("sequence exists")
        self.tables[seq_id] = []
        self.lens[seq_id] = 0

    def _blocks_needed(self, seq_id: int, n: int) -> int:
        bs = self.block_size
        L = self.lens[seq_id]
        tab = self.tables[seq_id]
        need = 0
        if n > 0 and L % bs != 0 and self.ref[tab[-1]] > 1:
            need += 1                                   # copy-on-write of the tail
        have_slots = len(tab) * bs - L
        extra = n - have_slots
        if extra > 0:
            need += (extra + bs - 1) // bs
        return need

    def _resident(self, seq_id: int) -> None:
        if seq_id not in self.tables:
            raise BlockManagerError("unknown sequence")
        if seq_id in self.swapped:
            raise BlockManagerError("sequence is swapped out")

    def append_tokens(self, seq_id: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Append n tokens; returns (slots, cow_pairs)."""
        self._resident(seq_id)
        if n < 0:
            raise BlockManagerError("negative count")
        if self._blocks_needed(seq_id, n) > self.available():
            raise OutOfBlocks()
        bs = self.block_size
        tab = self.tables[seq_id]
        slots: List[int] = []
        cow: List[Tuple[int, int]] = []
        for _ in range(n):
            L = self.lens[seq_id]
            if L % bs == 0 and L // bs == len(tab):
                tab.append(self._alloc())
            else:
                last = tab[L // bs]
                if self.ref[last] > 1:
                    fresh = self._alloc()
                    cow.append((last, fresh))
                    self._put(last)
                    tab[L // bs] = fresh
            slots.append(tab[L // bs] * bs + L % bs)
            self.lens[seq_id] = L + 1
        return slots, cow

    def make_private(self, seq_id: int, logical_block: int) -> List[Tuple[int, int]]:
        self._resident(seq_id)
        tab = self.tables[seq_id]
        b = tab[logical_block]
        if b < 0:
            raise BlockManagerError("block was released")
        if self.ref[b] <= 1:
            return []
        if self.available() < 1:
            raise OutOfBlocks()
        fresh = self._alloc()
        self._put(b)
        tab[logical_block] = fresh
        return [(b, fresh)]

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.tables:
            raise BlockManagerError("unknown parent")
        if parent in self.swapped:
            raise BlockManagerError("parent is swapped out")
        if child in self.tables:
            raise BlockManagerError("child exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            if b >= 0:
                self.ref[b] += 1

    def free_seq(self, seq_id: int) -> None:
        if seq_id not in self.tables:
            raise BlockManagerError("unknown sequence")
        for b in self.tables.pop(seq_id):
            if b >= 0:
                self._put(b)
        del self.lens[seq_id]
        self.swapped.pop(seq_id, None)

    def swap_out(self, seq_id: int) -> List[int]:
        """Releases the private tail of the table; returns its blocks."""
        self._resident(seq_id)
        tab = self.tables[seq_id]
        k = len(tab)
        while k > 0 and tab[k - 1] >= 0 and self.ref[tab[k - 1]] == 1:
            k -= 1
        out = tab[k:]
        for b in out:
            self._put(b)
        del tab[k:]
        self.swapped[seq_id] = len(out)
        return out

    def swap_in(self, seq_id: int) -> List[int]:
        """Re-allocates the swapped-out tail (all-or-nothing); returns the
        new blocks in logical order."""
        if seq_id not in self.swapped:
            raise BlockManagerError("sequence is not swapped out")
        n = self.swapped[seq_id]
        if n > self.available():
            raise OutOfBlocks()
        new = [self._alloc() for _ in range(n)]
        self.tables[seq_id].extend(new)
        del self.swapped[seq_id]
        return new

    def release_before(self, seq_id: int, first_pos: int) -> List[int]:
        """Drops the blocks wholly before logical position first_pos; returns
        the dropped table entries (block ids), in logical order."""
        self._resident(seq_id)
        tab = self.tables[seq_id]
        bs = self.block_size
        first_pos = min(max(int(first_pos), 0), self.lens[seq_id])
        dropped = []
        for j in range(min(first_pos // bs, len(tab))):
            if tab[j] >= 0:
                dropped.append(tab[j])
                self._put(tab[j])
                tab[j] = -1
        return dropped

    # -- prefix cache --------------------------------------------------------
    def cache_full_blocks(self, seq_id: int, tokens: Sequence[int]) -> int:
        """Registers the sequence's full blocks under their token prefixes;
        returns how many entries were added. ``tokens`` are the sequence's
        token ids from position 0 (at least as many as its full blocks)."""
        self._resident(seq_id)
        bs = self.block_size
        tab = self.tables[seq_id]
        n_full = min(self.lens[seq_id], len(tokens)) // bs
        added = 0
        for j in range(n_full):
            if tab[j] < 0:
                continue                                 # released by a window
            key = tuple(int(t) for t in tokens[:(j + 1) * bs])
            if key in self.cache:
                continue
            self.cache[key] = tab[j]
            self.ref[tab[j]] += 1
            added += 1
        return added

    def lookup(self, tokens: Sequence[int]) -> List[int]:
        """Blocks of the longest cached prefix of whole blocks (no LRU update)."""
        bs = self.block_size
        blocks = []
        for j in range(len(tokens) // bs):
            b = self.cache.get(tuple(int(t) for t in tokens[:(j + 1) * bs]))
            if b is None:
                break
            blocks.append(b)
        return blocks

    def add_seq_cached(self, seq_id: int, tokens: Sequence[int]) -> int:
        """Starts a sequence on the longest cached prefix of ``tokens``;
        returns the number of tokens it already holds."""
        if seq_id in self.tables:
            raise BlockManagerError("sequence exists")
        bs = self.block_size
        blocks = self.lookup(tokens)
        for j, b in enumerate(blocks):
            self.cache.move_to_end(tuple(int(t) for t in tokens[:(j + 1) * bs]))
            self.ref[b] += 1
        self.tables[seq_id] = list(blocks)
        self.lens[seq_id] = len(blocks) * bs
        return len(blocks) * bs

    def num_cached(self) -> int:
        return len(self.cache)

    # -- queries -----------------------------------------------------------
    def block_table(self, seq_id: int) -> List[int]:
        return list(self.tables[seq_id])

    def seq_len(self, seq_id: int) -> int:
        return self.lens[seq_id]

    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def check_invariants(self) -> None:
        """Sum of refcounts == sum of table lengths; a block is free iff its
        refcount is 0; every table covers exactly ceil(len / bs) blocks."""
        total_refs = sum(self.ref)
        total_entries = (sum(sum(1 for b in t if b >= 0) for t in self.tables.values())
                         + len(self.cache))
        assert total_refs == total_entries, (total_refs, total_entries)
        free = set(self.free)
        assert len(free) == len(self.free), "duplicate free entry"
        for b, r in enumerate(self.ref):
            assert (r == 0) == (b in free), (b, r)
        bs = self.block_size
        for s, t in self.tables.items():
            assert len(t) + self.swapped.get(s, 0) == (self.lens[s] + bs - 1) // bs
