"""ctypes declarations of libpagedkv.so (include/pagedkv.h).

The library is loaded from this package's directory only; if it is missing the
caller gets an error telling it to build (there is no fallback path).
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_WORKSPACE = -3
PA_ERR_CUDA = -4
PA_ERR_DEVICE = -5
PA_ERR_OOM = -6
PA_ERR_REFCOUNT = -7
PA_ERR_CAPACITY = -8

PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_SLOT = 2
PA_DEVERR_TIMEOUT = 4
PA_DEVERR_PAIR = 8
PA_DEVERR_CONTEXT = 16
PA_DEVERR_LAYOUT = 32
PA_DEVERR_RANGE = 64
PA_DEVERR_PLAN = 128

vp = C.c_void_p
i32 = C.c_int
i64 = C.c_int64
p_i32 = C.POINTER(C.c_int32)
p_i64 = C.POINTER(C.c_int64)

# name -> (restype, argtypes); every symbol declared in include/pagedkv.h
SIGNATURES = {
    "pa_decode_workspace_bytes": (C.c_size_t, [i32, i32, i32, i32, i32]),
    "pa_decode_partition_tokens": (i32, [i32, i32, i32, i32, i32, i32, i32]),
    "pa_decode": (i32, [vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32, i32,
                        vp, C.c_size_t, vp]),
    "pa_decode_ex": (i32, [vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32, i32,
                           i32, vp, C.c_size_t, vp]),
    "pa_decode_tc": (i32, [vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32, i32,
                           i32, vp, C.c_size_t, vp]),
    "pa_decode_noalloc": (i32, [vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32,
                                i32, vp]),
    "pa_reshape_and_cache": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
    "pa_copy_blocks": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp]),
    "pa_copy_blocks_ex": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
    "pa_decode_window": (i32, [vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32, i32,
                               i32, i32, vp, C.c_size_t, vp]),
    "pa_swap_out_blocks": (i32, [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, vp]),
    "pa_swap_in_blocks": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
    "pa_reshape_and_cache_fp8": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
    "pa_decode_fp8": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32,
                            i32, i32, vp, C.c_size_t, vp]),
    "pa_decode_plan": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, i32]),
    "pa_decode_planned": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32, i32,
                                i32, i32, i32, vp, i32, vp, C.c_size_t, vp]),
    "pa_prefill_paged": (i32, [vp, vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32,
                               i32, i32, vp]),
    "pa_prefill_workspace_bytes": (C.c_size_t, [i32, i32, i32, i32, i32]),
    "pa_prefill_paged_ex": (i32, [vp, vp, vp, vp, vp, vp, vp, C.c_float, i32, i32, i32, i32, i32, i32,
                                  i32, i32, i32, vp, C.c_size_t, vp]),
    "pa_get_device_error": (i32, [C.POINTER(C.c_int)]),
    "pa_selftest_wait_timeout": (i32, [i32, vp]),
    "pa_status_string": (C.c_char_p, [i32]),
    "pa_bm_create": (vp, [i32, i32]),
    "pa_bm_destroy": (None, [vp]),
    "pa_bm_add_seq": (i32, [vp, i64]),
    "pa_bm_append_tokens": (i32, [vp, i64, i32, p_i64, p_i64, i32, C.POINTER(C.c_int)]),
    "pa_bm_make_private": (i32, [vp, i64, i32, p_i64, C.POINTER(C.c_int)]),
    "pa_bm_fork": (i32, [vp, i64, i64]),
    "pa_bm_free_seq": (i32, [vp, i64]),
    "pa_bm_release_before": (i32, [vp, i64, i64, C.POINTER(C.c_int)]),
    "pa_bm_swap_out": (i32, [vp, i64, p_i32, i32, C.POINTER(C.c_int)]),
    "pa_bm_swap_in": (i32, [vp, i64, p_i32, i32, C.POINTER(C.c_int)]),
    "pa_bm_cache_blocks": (i32, [vp, i64, p_i32, i64, C.POINTER(C.c_int)]),
    "pa_bm_add_seq_cached": (i32, [vp, i64, p_i32, i64, p_i64]),
    "pa_bm_num_cached": (i32, [vp]),
    "pa_bm_block_table": (i32, [vp, i64, p_i32, i32, C.POINTER(C.c_int)]),
    "pa_bm_seq_len": (i64, [vp, i64]),
    "pa_bm_num_free": (i32, [vp]),
    "pa_bm_refcount": (i32, [vp, i32]),
    "pa_bm_build_batch": (i32, [vp, p_i64, i32, i32, p_i32, p_i32]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Loads the library (once) and declares every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python paged_kv_cache_59_gb300/build.py`")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = load().pa_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} ({status})")


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedKVError(fn, status)
