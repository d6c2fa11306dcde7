"""fp8 (E4M3) KV cache, oracle side: decode, encode, cache write, attention.

Test infrastructure (see the package header): only tests, the smoke check and
the benchmark's CPU legs use it.

Sources (cited by page title and section):
* "Inference serving: the KV-cache machine", section "What insiders know":
  an fp8 KV cache holds twice the tokens in the same pool; the hard part is
  the scale factors, kept per head (or finer) because outlier magnitudes
  live in particular heads.
* "KV Cache Explained Like You're an LLM Engineer", section "Future
  Optimizations" / "KV Cache Quantization": one byte per cached element with
  a scale; dequantisation is code * scale.
* "Modern AI Infrastructure and Agentic System Design", 9.1 "High-Throughput
  Model Serving Architectures", part "Quantization and speculative
  decoding": decode is bandwidth bound, so fewer bytes per cached element cut
  the time to read the cache in proportion.

The E4M3 format (the 8-bit floating-point definition with 4 exponent bits,
3 mantissa bits, exponent bias 7 and no infinities): sign s, exponent field
e, mantissa field m;
  e = 0          -> (-1)^s * (m / 8) * 2^-6          (zero and subnormals)
  0 < e < 15, or e = 15 with m < 7
                 -> (-1)^s * (1 + m / 8) * 2^(e - 7)  (largest: 448)
  e = 15, m = 7  -> NaN.

Readings taken where the pages are silent:
* Scales: one fp32 scale per KV head for K and one for V, given as inputs
  (calibrated offline in practice). A cached element stands for
  decode(code) * scale.
* Encoding of a new element x (bf16): the quotient x / scale is formed in
  fp32 (IEEE division, round to nearest even), because that is the precision
  in which the kernel decides the code. It is then rounded to the nearest
  E4M3 value, ties to the even mantissa. Finite values beyond the largest
  magnitude saturate to +-448, and infinities do too. The sign of a zero
  result is kept; NaN becomes 0x7F.
* Attention over an fp8 cache is the plain definition applied to the
  dequantised values (``attention.attend``), in fp64.
"""
from __future__ import annotations

import numpy as np

from . import attention
from .bf16 import bf16_bits_to_f64

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of each E4M3 code (uint8 array) as fp64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * mag
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)


# the 127 non-negative finite values, in code order (which is increasing)
_POS_VALUES = e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))


def f64_to_e4m3(x) -> np.ndarray:
    """Round fp64 values to E4M3 codes: nearest, ties to even mantissa,
    saturating at +-448 (infinities included), NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(nan, E4M3_NAN_CODE, code)
    return code.astype(np.uint8)


def quantize(x_bf16_bits, scale) -> np.ndarray:
    """E4M3 codes of bf16 values x (bits, [..., D]) for the given fp32 scale
    (broadcast against x): code = round_e4m3(fp32(x) / fp32(scale))."""
    x32 = bf16_bits_to_f64(x_bf16_bits).astype(np.float32)  # exact
    q32 = x32 / np.asarray(scale, dtype=np.float32)          # one IEEE fp32 division
    return f64_to_e4m3(q32.astype(np.float64))


def reshape_and_cache_fp8(k_new, v_new, k_pool8, v_pool8, slot_mapping, k_scale, v_scale):
    """The cache write for an fp8 cache.

    k_new, v_new bf16 bits [T][n_kv_heads][head_dim]; pools uint8
    [blocks][n_kv_heads][bs][head_dim]; k_scale, v_scale fp32 [n_kv_heads].
    Row t goes to (block, offset) = divmod(slot_mapping[t], bs) for every KV
    head, head h encoded with its own scale; rows with a negative slot are
    skipped. Returns new pools (the inputs are not modified).
    """
    kp = np.array(k_pool8, copy=True)
    vp = np.array(v_pool8, copy=True)
    bs = kp.shape[2]
    ks = np.asarray(k_scale, dtype=np.float32)[:, None]
    vs = np.asarray(v_scale, dtype=np.float32)[:, None]
    for t, s in enumerate(np.asarray(slot_mapping)):
        if int(s) < 0:
            continue
        blk, off = int(s) // bs, int(s) % bs
        kp[blk, :, off, :] = quantize(np.asarray(k_new)[t], ks)
        vp[blk, :, off, :] = quantize(np.asarray(v_new)[t], vs)
    return kp, vp


def dequantize(codes, scale) -> np.ndarray:
    """decode(code) * scale in fp64 (scale broadcast against codes)."""
    return e4m3_to_f64(codes) * np.asarray(scale, dtype=np.float64)


def _seq_kv(k_pool8, v_pool8, table_row, n, kvh, k_scale, v_scale):
    kc = attention.gather_kv(np.asarray(k_pool8)[:, kvh:kvh + 1], table_row, n)[:, 0, :]
    vc = attention.gather_kv(np.asarray(v_pool8)[:, kvh:kvh + 1], table_row, n)[:, 0, :]
    return dequantize(kc, float(np.float32(k_scale[kvh]))), dequantize(vc, float(np.float32(v_scale[kvh])))


def paged_decode_fp8(q, k_pool8, v_pool8, block_tables, context_lens, scale, k_scale, v_scale):
    """Single-query attention of every sequence over its fp8 paged cache.

    q bf16 bits [B][H][D]; returns fp64 [B][H][D]; ctx <= 0 gives a zero row.
    """
    q = np.asarray(q)
    B, H, D = q.shape
    Hk = np.asarray(k_pool8).shape[1]
    g = H // Hk
    out = np.zeros((B, H, D), dtype=np.float64)
    for b in range(B):
        n = int(context_lens[b])
        if n <= 0:
            continue
        for kvh in range(Hk):
            kc, vc = _seq_kv(k_pool8, v_pool8, block_tables[b], n, kvh, k_scale, v_scale)
            for h in range(kvh * g, (kvh + 1) * g):
                out[b, h] = attention.attend(q[b, h], kc, vc, scale)
    return out


def paged_decode_fp8_rows(q, k_pool8, v_pool8, block_tables, context_lens, scale, k_scale, v_scale,
                          rows):
    """paged_decode_fp8 for a subset of (seq, head) pairs; {(b, h): out[D]}."""
    q = np.asarray(q)
    H = q.shape[1]
    Hk = np.asarray(k_pool8).shape[1]
    g = H // Hk
    res, cache = {}, {}
    for b, h in rows:
        b, h = int(b), int(h)
        n = int(context_lens[b])
        if n <= 0:
            res[(b, h)] = np.zeros(q.shape[2])
            continue
        key = (b, h // g)
        if key not in cache:
            cache[key] = _seq_kv(k_pool8, v_pool8, block_tables[b], n, h // g, k_scale, v_scale)
        kc, vc = cache[key]
        res[(b, h)] = attention.attend(q[b, h], kc, vc, scale)
    return res
