"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of the oracle (a dropped
scale, a wrong index, an off-by-one causal bound, a tie rounded the wrong
way, a block freed too early, ...) and runs the pin tests of that module
against the copy. Every mutant must fail at least one pin; a mutant that
survives means the pins do not pin the oracle. The mistake is planted on the
CPU, in a temporary copy; the repository's oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

from tests.conftest import ROOT

MUTANTS = [
    # (oracle file, pin tests, original text, mutated text, what the mistake is)
    ("attention.py", "test_oracle_attention.py", "kh = h // g", "kh = h % Hk", "wrong GQA head map"),
    ("attention.py", "test_oracle_attention.py", "s = (k @ q) * float(scale)", "s = (k @ q)", "dropped scale"),
    ("attention.py", "test_oracle_attention.py", "return (p @ v) / p.sum()", "return (p @ k) / p.sum()",
     "K in place of V"),
    ("attention.py", "test_oracle_attention.py",
     "out[t] = pool[int(table_row[t // bs]), :, t % bs, :]",
     "out[t] = pool[int(table_row[t // bs]), :, (t + 1) % bs, :]", "off-by-one slot in the gather"),
    ("attention.py", "test_oracle_attention.py", "kc[:p + 1, kh, :], vc[:p + 1, kh, :]",
     "kc[:p, kh, :], vc[:p, kh, :]", "off-by-one causal bound"),
    ("attention.py", "test_oracle_attention.py", "p = n - L + i", "p = n - L + i - 1", "shifted chunk position"),
    ("attention.py", "test_oracle_attention.py", "p = np.exp(s - s.max())", "p = np.exp(s)",
     "no maximum subtraction"),
    ("fp8.py", "test_oracle_fp8.py", "((d_hi == d_lo) & (hi % 2 == 0))", "((d_hi == d_lo) & (hi % 2 == 1))",
     "ties to odd"),
    ("fp8.py", "test_oracle_fp8.py", "np.exp2(e.astype(np.float64) - 7.0)", "np.exp2(e.astype(np.float64) - 8.0)",
     "exponent bias off by one"),
    ("fp8.py", "test_oracle_fp8.py", "(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7", "subnormal scale"),
    ("fp8.py", "test_oracle_fp8.py", "q32 = x32 / np.asarray(scale, dtype=np.float32)",
     "q32 = x32 * np.asarray(scale, dtype=np.float32)", "scale multiplied instead of divided"),
    ("block_manager.py", "test_oracle_block_manager.py",
     "self.ref[b] -= 1\n        if self.ref[b] == 0:", "self.ref[b] -= 1\n        if self.ref[b] <= 1:",
     "block freed while still referenced"),
    ("attention.py", "test_oracle_window.py", "lo = max(0, n - 1 - int(window))",
     "lo = max(0, n - int(window))", "window one position short"),
    ("cache_ops.py", "test_oracle_cache_and_sizes.py", "kp[blk, :, off, :] = k_new[t]",
     "kp[blk, :, off, :] = v_new[t]", "V written into the K pool"),
    ("cache_ops.py", "test_oracle_cache_and_sizes.py", "kp[int(dst)] = kp[int(src)]",
     "kp[int(src)] = kp[int(dst)]", "block copied the wrong way"),
    ("block_manager.py", "test_oracle_block_manager.py", "if self.ref[last] > 1:", "if self.ref[last] > 2:",
     "write into a block shared by two tables"),
]


@pytest.mark.parametrize("fname,pins,old,new,what", MUTANTS, ids=[m[4] for m in MUTANTS])
def test_mutant_fails_a_pin(tmp_path, fname, pins, old, new, what):
    for d in ("oracle", "workloads", "tests"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("__pycache__", "*.so"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path / "pytest.ini")
    target = tmp_path / "oracle" / fname
    src = target.read_text()
    assert src.count(old) >= 1, f"the text to mutate ({what}) is no longer in oracle/{fname}"
    target.write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.join("tests", pins)],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 1, f"mutant survived ({what}):\n{r.stdout[-1500:]}"
