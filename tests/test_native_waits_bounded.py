"""Static check of the device code's waits.

Every wait in a kernel must end: a kernel that spins on a barrier nothing
completes would hang the GPU. The device code keeps all of its spinning in
two helpers that give up after a time limit (pa::mbar_wait, with a
%globaltimer limit, and the prefill's wait_bar, with a 1 s limit and an
abort flag). This test reads the native sources and checks that:

- the raw mbarrier polls (mbar_try_wait, mbar_try_wait_sleep) are called only
  inside those two helpers;
- every loop without a condition is one of the reviewed ones below, each of
  which ends for the reason given;
- every call of those helpers in a kernel is made with a result or a limit
  that is used (mbar_wait calls pass an error word or a limit).

A new unbounded loop or a raw poll elsewhere fails here, on the CPU, before
it can run on a GPU.
"""
import os
import re

from tests.conftest import ROOT

CSRC = os.path.join(ROOT, "paged_kv_cache_59_gb300", "csrc")

# (file, loop text) -> why it ends
REVIEWED_UNCONDITIONAL_LOOPS = {
    ("pa_common.cuh", "for (uint32_t it = 1;; ++it) {"): "mbar_wait: returns once the %globaltimer limit passes",
    ("prefill.cu", "for (uint32_t it = 1;; ++it) {"): "wait_bar: returns after 1 s or once another role aborted",
    ("prefill.cu", "for (int seg = 0;; ++seg) {"): "segment loop: breaks when the work-list counter passes its "
                                                   "end (balanced) or after one segment (per pair)",
}


def _sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".cpp")):
            src = open(os.path.join(CSRC, f)).read()
            out[f] = re.sub(r"//[^\n]*", "", src)  # comments removed, lines kept
    return out


def _enclosing_function(src, pos):
    """Name of the function whose body contains offset pos (by brace depth)."""
    depth, i = 0, pos
    while i > 0:
        i -= 1
        c = src[i]
        if c == "}":
            depth += 1
        elif c == "{":
            if depth == 0:
                head = src[max(0, i - 400):i]
                m = re.findall(r"([A-Za-z_]\w*)\s*\([^;{}]*\)\s*(?:const\s*)?$", head.rstrip())
                if m:
                    return m[-1]
            else:
                depth -= 1
    return None


def test_raw_polls_only_inside_the_bounded_helpers():
    allowed = {("pa_common.cuh", "mbar_wait"), ("prefill.cu", "wait_bar")}
    for f, src in _sources().items():
        for m in re.finditer(r"\bmbar_try_wait(?:_sleep)?\s*\(", src):
            line_start = src.rfind("\n", 0, m.start()) + 1
            if re.match(r"\s*__device__", src[line_start:m.start()]):  # the poll's own definition
                continue
            fn = _enclosing_function(src, m.start())
            assert (f, fn) in allowed, f"{f}: raw mbarrier poll in {fn}"


def test_unconditional_loops_are_reviewed():
    found = set()
    for f, src in _sources().items():
        for m in re.finditer(r"for\s*\([^;)]*;\s*;[^)]*\)\s*\{|while\s*\(\s*(?:true|1)\s*\)\s*\{", src):
            found.add((f, re.sub(r"\s+", " ", m.group(0)).strip()))
    assert found == set(REVIEWED_UNCONDITIONAL_LOOPS), found ^ set(REVIEWED_UNCONDITIONAL_LOOPS)


def test_helpers_give_up():
    src = _sources()
    common = src["pa_common.cuh"]
    body = common[common.index("bool mbar_wait("):]
    body = body[:body.index("\n}\n")]
    assert "globaltimer_ns()" in body and "limit_ns" in body and "return false" in body
    pf = src["prefill.cu"]
    body = pf[pf.index("bool wait_bar("):]
    body = body[:body.index("\n}\n")]
    assert "PA_WAIT_LIMIT_NS" in body and "abort_flag" in body and "return false" in body


def _loop_body(src, start):
    """Body text of the loop whose header starts at offset `start`."""
    i = src.index("{", start)
    depth = 0
    for k in range(i, len(src)):
        if src[k] == "{":
            depth += 1
        elif src[k] == "}":
            depth -= 1
            if depth == 0:
                return src[i + 1:k]
    raise AssertionError("unbalanced braces")


def _without_lambdas(body):
    """The text with every lambda's body removed (a return there leaves the
    lambda, not the loop)."""
    out, i = [], 0
    for m in re.finditer(r"\[[&=]?\]\s*\(", body):
        if m.start() < i:
            continue
        k, depth = m.end() - 1, 0          # the parameter list, parentheses balanced
        while True:
            depth += {"(": 1, ")": -1}.get(body[k], 0)
            k += 1
            if depth == 0:
                break
        k = body.index("{", k)
        out.append(body[i:k])
        depth = 0                          # the body, braces balanced
        while True:
            depth += {"{": 1, "}": -1}.get(body[k], 0)
            k += 1
            if depth == 0:
                break
        i = k
    out.append(body[i:])
    return "".join(out)


def test_named_barrier_arrivals_and_syncs_balance():
    """The prefill hands each tile's P to the MMA warp through a hardware named
    barrier, which has no time limit. It cannot be left waiting because each
    side meets it exactly once per key tile: the arrive and the syncs sit in
    loops `for (int j = 0; j < n_kt; ++j)` with no break, continue or return
    (a failed mbarrier wait only stops the waiting, not the loop)."""
    pf = _sources()["prefill.cu"]
    uses = [m.start() for m in re.finditer(r"bar\.(sync|arrive) ", pf)]
    assert uses, "no named barrier found"
    loops = [m.start() for m in re.finditer(r"for \(int j = 0; j < n_kt; \+\+j\) \{", pf)]
    covered = 0
    for start in loops:
        body = _loop_body(pf, start)
        n_bar = len(re.findall(r"bar\.(?:sync|arrive) ", body))
        if not n_bar:
            continue
        covered += n_bar
        assert not re.search(r"\b(break|continue|return)\b", _without_lambdas(body)), \
            "a loop with a named barrier can exit early"
    assert covered == len(uses), "a named barrier outside the per-key-tile loops"
    arrives = re.findall(r'bar\.arrive %0, (\d+);', pf)
    syncs = re.findall(r'bar\.sync (\d), (\d+);', pf)
    assert len(arrives) == 1 and sorted(i for i, _ in syncs) == ["1", "2"]
    assert all(c == arrives[0] for _, c in syncs)        # the same thread count on both sides
    assert int(arrives[0]) == 4 * 32 + 32                # four softmax warps arrive, one warp syncs
