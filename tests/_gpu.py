"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import pytest

# Tolerance for bf16 attention outputs against the fp64 oracle, applied per
# element: |gpu - ref| <= ATOL + RTOL * |ref| (max-abs 2e-3, max-rel 1e-2).
ATOL = 2e-3
RTOL = 1e-2


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(x: np.ndarray):
    """numpy -> CUDA tensor; uint16 (bf16 bits) travels as int16."""
    torch = torch_cuda()
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host_bits(t) -> np.ndarray:
    """CUDA bf16/int16 tensor -> numpy uint16 bits."""
    torch = torch_cuda()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    # decoding only (widening is exact); independent of the oracle module
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# Every comparison's error figures, for the session summary printed by
# tests/conftest.py: per test, the number of outputs compared, the largest
# absolute error, the largest relative error over |ref| > 1e-2, and the
# largest ratio of error to the element-wise bound.
PARITY_STATS = {}


def _record(what: str, n: int, max_abs: float, max_rel: float, worst_frac: float) -> None:
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", what).split(" ")[0]
    s = PARITY_STATS.setdefault(test, {"n": 0, "max_abs": 0.0, "max_rel": 0.0, "bound_frac": 0.0})
    s["n"] += n
    s["max_abs"] = max(s["max_abs"], max_abs)
    s["max_rel"] = max(s["max_rel"], max_rel)
    s["bound_frac"] = max(s["bound_frac"], worst_frac)


def assert_attention_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    got = bf16_to_f64(gpu_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; worst at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r}")
    big = np.abs(ref) > 1e-2
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "max_rel": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
             "bound_frac": float((err / bound).max()) if err.size else 0.0}
    _record(what, int(err.size), stats["max_abs"], stats["max_rel"], stats["bound_frac"])
    return stats


def check_device_error(expected: int = 0) -> None:
    import paged_kv_cache_59_gb300 as pk
    flags = pk.pa_get_device_error()
    assert flags == expected, f"device error word {flags:#x}, expected {expected:#x}"
