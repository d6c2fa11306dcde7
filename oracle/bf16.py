"""Exact bf16 -> fp64 decoding (oracle side).

A bf16 value is the upper 16 bits of an IEEE fp32; widening to fp32 and then
to fp64 is exact, so the oracle treats the stored bf16 inputs as exact numbers.
"""
import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
