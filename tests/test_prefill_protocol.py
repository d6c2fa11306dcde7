"""A discrete-event model of the prefill kernel's barrier protocol.

The chunked-prefill kernel runs five roles: a TMA producer (K and V tiles
into kKS and kVS shared-memory stages), four converter warps (each landed V
tile rewritten in place), one MMA-issuing thread (QK and PV for two query
tiles A and B, issued in order into one tensor-core pipe), and two softmax
warpgroups of four warps. They meet on mbarriers, except for the hand-over
of a tile's P, where the four softmax warps arrive on a named barrier and
the MMA warp syncs on it. This model replays the same waits and arrivals
with random delays and checks, for every schedule it draws:

- every parity wait targets phase c or c + 1 of its barrier, where c phases
  have completed, so the wait's parity names exactly one phase;
- the run finishes (no deadlock);
- each QK reads the K tile it names and each PV the V tile it names, and that
  tile has been converted; a converter finishes a tile before the next load
  lands in its stage;
- a softmax warpgroup that rescales O at step j finds P.V of step j-1 done
  (it waits for no barrier of its own: S(j) is issued after that P.V);
- no softmax warp arrives on a tile's named barrier for step j+1 before the
  MMA warp has synced for step j (a hardware barrier has no phases).

The stage counts are read from the kernel source, so the model follows them.
A mutated protocol (PV_A waiting for the landed V tile instead of the
converted one) must fail, which shows the checks have teeth.
"""
import os
import random
import re

import pytest

from tests.conftest import ROOT


def _stage_counts():
    src = open(os.path.join(ROOT, "paged_kv_cache_59_gb300", "csrc", "prefill.cu")).read()
    ks = int(re.search(r"constexpr int kKS = (\d+);", src).group(1))
    vs = int(re.search(r"constexpr int kVS = (\d+);", src).group(1))
    return ks, vs


class Bar:
    def __init__(self, name, count=1):
        self.name, self.count, self.pending, self.c = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, self.name
        if self.pending == 0:
            self.c += 1
            self.pending = self.count


def run(n, KS, VS, seed, pv_waits_converter=True):
    rng = random.Random(seed)
    k_full = [Bar(f"k_full{i}") for i in range(KS)]
    k_free = [Bar(f"k_free{i}") for i in range(KS)]
    v_full = [Bar(f"v_full{i}") for i in range(VS)]
    v_free = [Bar(f"v_free{i}") for i in range(VS)]
    v_conv = [Bar(f"v_conv{i}", 4) for i in range(VS)]
    s_full = [Bar("s_full0"), Bar("s_full1")]
    p_named = [Bar("named0", 4), Bar("named1", 4)]  # four softmax warps arrive; the MMA warp syncs
    synced = [0, 0]                                   # steps the MMA warp has synced per tile
    pv_done = [Bar("pv_done0"), Bar("pv_done1")]
    done_ops = set()
    pipe, tma = [], []
    kslot, vslot, vconv_of = {}, {}, {}  # stage -> tile landed / tile converted there

    def wait(bar, k):  # parity wait for phase k (k counts from 0)
        def cond():
            assert bar.c in (k, k + 1), f"{bar.name}: wait for phase {k} with {bar.c} complete"
            return bar.c == k + 1
        return cond

    def idle(m):
        for _ in range(m):
            yield lambda: True

    def producer():
        nk = nv = 0
        while nk < min(KS, n):
            tma.append(("k", nk, rng.randint(1, 40))); nk += 1
        while nv < min(VS, n):
            tma.append(("v", nv, rng.randint(1, 40))); nv += 1
        while nk < n or nv < n:
            if nk < n and nk <= nv:
                yield wait(k_free[nk % KS], (nk - KS) // KS)
                tma.append(("k", nk, rng.randint(1, 40))); nk += 1
            else:
                yield wait(v_free[nv % VS], (nv - VS) // VS)
                tma.append(("v", nv, rng.randint(1, 40))); nv += 1
            yield from idle(rng.choice([0, 0, 5, 80]))

    def converter(w):
        for j in range(n):
            yield wait(v_full[j % VS], j // VS)
            for _ in range(rng.randint(1, 12)):  # rewriting the stage in place
                assert vslot.get(j % VS) == j, f"V({j}) overwritten while converter {w} works on it"
                yield lambda: True
            if w == 0:
                vconv_of[j % VS] = j
            v_conv[j % VS].arrive()

    def mma():
        yield wait(k_full[0], 0)
        pipe.append(([s_full[0]], ("qk", 0, 0)))
        pipe.append(([s_full[1], k_free[0]], ("qk", 1, 0)))
        for j in range(n):
            if pv_waits_converter:
                yield wait(v_conv[j % VS], j // VS)
            else:
                yield wait(v_full[j % VS], j // VS)
            if j + 1 < n:
                yield wait(k_full[(j + 1) % KS], (j + 1) // KS)
            yield wait(p_named[0], j)
            synced[0] = j + 1
            pipe.append(([pv_done[0]], ("pv", 0, j)))
            if j + 1 < n:
                pipe.append(([s_full[0]], ("qk", 0, j + 1)))
            yield wait(p_named[1], j)
            synced[1] = j + 1
            pipe.append(([v_free[j % VS], pv_done[1]], ("pv", 1, j)))
            if j + 1 < n:
                pipe.append(([k_free[(j + 1) % KS], s_full[1]], ("qk", 1, j + 1)))

    def softmax(x):
        for j in range(n):
            yield wait(s_full[x], j)
            if j > 0:  # an O rescale here would need P.V of step j-1 done
                assert ("pv", x, j - 1) in done_ops, f"softmax {x} step {j}: PV({j - 1}) not done"
            yield from idle(rng.randint(0, 5))
            assert synced[x] >= j, f"tile {x}: arrival for step {j} before the sync of step {j - 1}"
            p_named[x].arrive()
        yield wait(pv_done[x], n - 1)

    actors = [producer(), mma()] + [converter(w) for w in range(4)] + [softmax(x) for x in (0, 1) for _ in range(4)]
    conds = [None] * len(actors)
    done = [False] * len(actors)
    busy = 0
    for _ in range(10 ** 6):
        if all(done):
            return
        for i in range(len(tma) - 1, -1, -1):
            kind, j, t = tma[i]
            if t > 1:
                tma[i] = (kind, j, t - 1)
                continue
            tma.pop(i)
            if kind == "k":
                kslot[j % KS] = j
                k_full[j % KS].arrive()
            else:
                vslot[j % VS] = j
                v_full[j % VS].arrive()
        if pipe:
            if busy <= 0:
                busy = rng.randint(1, 20)
            busy -= 1
            if busy <= 0:
                bars, (op, x, j) = pipe.pop(0)
                if op == "qk":
                    assert kslot.get(j % KS) == j, f"QK{x}({j}) read the wrong K tile"
                else:
                    assert vslot.get(j % VS) == j, f"PV{x}({j}) read the wrong V tile"
                    assert vconv_of.get(j % VS) == j, f"PV{x}({j}) read V before it was converted"
                done_ops.add((op, x, j))
                for b in bars:
                    b.arrive()
        order = list(range(len(actors)))
        rng.shuffle(order)
        progressed = False
        for a in order:
            if done[a] or (conds[a] is not None and not conds[a]()):
                continue
            try:
                conds[a] = next(actors[a])
            except StopIteration:
                done[a] = True
            progressed = True
        assert progressed or tma or pipe, "deadlock"
    raise AssertionError("no progress")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 17, 40])
def test_protocol_holds_under_random_schedules(n):
    ks, vs = _stage_counts()
    for seed in range(60):
        run(n, ks, vs, seed)


def test_mutated_protocol_is_caught():
    """PV_A waiting for the landed V tile rather than the converted one must
    fail some schedule."""
    ks, vs = _stage_counts()
    failures = 0
    for seed in range(200):
        try:
            run(6, ks, vs, seed, pv_waits_converter=False)
        except AssertionError:
            failures += 1
    assert failures > 0
