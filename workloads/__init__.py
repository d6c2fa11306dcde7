"""Seeded synthetic inputs for the paged-KV decode, cache-write, block-copy and
chunked-prefill workloads.

This package is shared by the fp64 oracle's tests, the CUDA path's tests and the
benchmark. It only draws numbers and lays them out: it contains no attention,
softmax or reduction arithmetic. Values are drawn N(0, 1) in fp32 and rounded
to bf16 (round to nearest even); bf16 tensors are carried as uint16 bit
patterns so that numpy, torch and the C ABI all see the same bytes.
"""
from .generate import (  # noqa: F401
    BLOCK_SIZE,
    BF16_NAN,
    Workload,
    WORKLOADS,
    make_workload,
    make_decode_case,
    make_prefill_case,
    f32_to_bf16_bits,
)
