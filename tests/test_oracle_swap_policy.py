"""Pin of the block manager's preemption by swapping: the simulator run of
"Inference serving: the KV-cache machine" (Lab B) is restated here as a
driver over this package's block manager (the Python model and the C++
manager), and must reproduce every number the page prints for it
(tests/golden/paged_sim_lab_b.txt).

The driver is this file's own restatement of the lab's policy, step for
step (the order of admission, swap-in and the decode iteration decides the
counts): one shared prompt table that every request forks; per iteration,
admit while a block is free and fewer than 256 are resident, swap in the
oldest preempted request while its private blocks fit, then advance every
resident by one token, preempting (swap_out) the resident with the most
tokens when a block is needed and none is free.
"""
import math
import random

import pytest

from oracle.block_manager import BlockManagerModel
from tests.conftest import read_golden

BS, PROMPT, POOL, NREQ, MAX_RESIDENT = 16, 512, 3072, 400, 256
ROOT = 10 ** 6


def chat_lengths(n, seed=7):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        r = rng.random()
        if r < 0.60:
            out.append(rng.randint(32, 200))
        elif r < 0.90:
            out.append(rng.randint(200, 700))
        else:
            out.append(rng.randint(700, 2000))
    return out


def run(m):
    lens = chat_lengths(NREQ)
    m.add_seq(ROOT)
    m.append_tokens(ROOT, PROMPT)                 # the one copy of the shared prompt
    prompt_blocks = list(m.block_table(ROOT))
    tok = {}
    running, swapped, waiting = [], [], list(range(NREQ))
    swaps = iters = peak = peak_blocks = 0
    while waiting or running or swapped:
        while waiting and m.num_free() >= 1 and len(running) < MAX_RESIDENT:
            r = waiting.pop(0)
            m.fork(ROOT, r)                       # aliases the prompt's blocks
            tok[r] = PROMPT
            running.append(r)
        while swapped and m.num_free() >= math.ceil(tok[swapped[0]] / BS) - PROMPT // BS:
            v = swapped.pop(0)
            m.swap_in(v)
            running.append(v)
        for s in list(running):
            if s not in running:                  # preempted earlier in this iteration
                continue
            if tok[s] % BS == 0 and m.num_free() == 0:
                v = max(running, key=lambda x: tok[x])
                m.swap_out(v)
                running.remove(v)
                swapped.append(v)
                swaps += 1
                continue
            m.append_tokens(s, 1)
            tok[s] += 1
            if tok[s] >= PROMPT + lens[s]:
                m.free_seq(s)
                running.remove(s)
        iters += 1
        peak = max(peak, len(running))
        peak_blocks = max(peak_blocks, POOL - m.num_free())
    return {"mean_gen": round(sum(lens) / NREQ), "peak_resident": peak, "peak_blocks": peak_blocks,
            "iterations": iters, "swaps": swaps, "prompt_blocks": len(prompt_blocks),
            "prompt_refcount_at_end": m.refcount(prompt_blocks[0]),
            "cow_blocks_saved": (NREQ - 1) * len(prompt_blocks)}


def expected():
    return {k: int(v) for k, v in read_golden("paged_sim_lab_b.txt")}


def test_model_reproduces_the_printed_run():
    assert run(BlockManagerModel(POOL, BS)) == expected()


def test_cpp_manager_reproduces_the_printed_run(capi):
    from paged_kv_cache_59_gb300 import BlockManager
    assert run(BlockManager(POOL, BS)) == expected()


def test_swap_round_trip_restores_the_table_shape():
    m = BlockManagerModel(20, BS)
    m.add_seq(0)
    m.append_tokens(0, 40)                        # 3 blocks
    m.fork(0, 1)
    m.append_tokens(1, 30)                        # child: block 2 copied (CoW) + 2 new
    out = m.swap_out(1)
    assert len(out) == 3                          # the child's private tail
    assert m.block_table(1) == m.block_table(0)[:2]
    assert m.seq_len(1) == 70
    m.check_invariants()
    new = m.swap_in(1)
    assert len(new) == 3 and m.block_table(1)[2:] == new
    m.append_tokens(1, 1)
    m.check_invariants()
