import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden(name: str):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    rows = []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def capi():
    """The built C-ABI library (built in-tree on first use)."""
    from paged_kv_cache_59_gb300 import build as _b
    from paged_kv_cache_59_gb300 import _capi
    _b.build()
    return _capi.load()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Attention parity figures of the GPU tests (the tolerance is applied per
    element as |gpu - ref| <= 2e-3 + 1e-2 |ref|; the pair of maxima below is
    reported besides): outputs compared, max-abs over all of them, max-rel
    over |ref| > 1e-2, and the worst error as a fraction of its bound."""
    stats = sys.modules.get("tests._gpu")
    stats = getattr(stats, "PARITY_STATS", None) if stats else None
    if not stats:
        return
    n = sum(s["n"] for s in stats.values())
    worst_abs = max(stats.items(), key=lambda kv: kv[1]["max_abs"])
    worst_rel = max(stats.items(), key=lambda kv: kv[1]["max_rel"])
    worst_frac = max(stats.items(), key=lambda kv: kv[1]["bound_frac"])
    tr = terminalreporter
    tr.write_line(f"attention parity: {n} outputs in {len(stats)} tests; "
                  f"max-abs {worst_abs[1]['max_abs']:.3e} ({worst_abs[0].split('::')[-1]}); "
                  f"max-rel(|ref|>1e-2) {worst_rel[1]['max_rel']:.3e} ({worst_rel[0].split('::')[-1]}); "
                  f"worst err/bound {worst_frac[1]['bound_frac']:.3f} ({worst_frac[0].split('::')[-1]})")
