"""Seeded synthetic inputs for the paged-KV decode, cache-write, block-copy and
chunked-prefill workloads.

This package is shared by the fp64 oracle's tests, the CUDA path's tests and the
benchmark. It only draws numbers and lays them out: it contains no attention,
softmax or reduction arithmetic. Values are drawn N(0, 1) in fp32 and rounded
to bf16 (round to nearest even); bf16 tensors are carried as uint16 bit
patterns so that numpy, torch and the C ABI all see the same bytes. An fp8
(E4M3) cache is drawn directly as random finite codes (uint8).
"""
from .generate import (  # noqa: F401
    BLOCK_SIZE,
    BF16_NAN,
    Workload,
    WORKLOADS,
    make_workload,
    make_decode_case,
    make_prefill_case,
    make_decode_case_fp8,
    make_decode_case_window,
    E4M3_NAN,
    f32_to_bf16_bits,
)
