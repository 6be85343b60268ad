"""ctypes view of libpagedattn.so (the C ABI declared in include/pa.h)."""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpagedattn.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_RANGE, PA_ERR_TIMEOUT, \
    PA_ERR_CUDA = range(6)
PA_BF16, PA_FP8_E4M3, PA_FP32 = 0, 1, 2
PA_WORKSPACE_HEADER_BYTES = 256
PA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_LENGTHS, PA_DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_OUT_OF_RANGE", 4: "PA_ERR_TIMEOUT", 5: "PA_ERR_CUDA"}

EXPORTED = ["pa_cache_append", "pa_attention_workspace_size", "pa_attention", "pa_check_error",
            "pa_workspace_init", "pa_last_error_string", "pa_version",
            "pa_set_kernel_timing_events", "pa_set_prefill_timing_events",
            "pa_attention_noalloc", "pa_copy_blocks", "pa_set_kernel_span_buffer",
            "pa_set_wait_limit_ns",
            "pa_test_skip_one_copy", "pa_selftest_wait_timeout"]
EXPORTED_BM = ["pa_bm_create", "pa_bm_destroy", "pa_bm_num_free", "pa_bm_append",
               "pa_bm_append_tokens", "pa_bm_fork", "pa_bm_free", "pa_bm_block_table",
               "pa_bm_num_tokens", "pa_bm_refcount", "pa_bm_cached_prefix"]


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_LIB = None


def load() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built (there is no fallback)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_286_gb300.build` "
            "(the paged-attention path has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64p, i32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p
    L.pa_cache_append.argtypes = [vp, vp, i64p, i32, vp, vp, ctypes.POINTER(CacheDesc), vp, vp]
    L.pa_cache_append.restype = ctypes.c_int
    L.pa_attention_workspace_size.argtypes = [i32] * 8
    L.pa_attention_workspace_size.restype = ctypes.c_size_t
    L.pa_attention.argtypes = [vp, i32, vp, vp, ctypes.POINTER(CacheDesc), i32p, i32, i32p, i32p,
                               i32, i32, i32, i32, i32, i32, ctypes.c_float, vp, i32, vp,
                               ctypes.c_size_t, vp]
    L.pa_attention.restype = ctypes.c_int
    L.pa_attention_noalloc.argtypes = [vp, i32, vp, vp, ctypes.POINTER(CacheDesc), i32p, i32,
                                       i32p, i32p, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                                       vp, i32, vp, vp]
    L.pa_attention_noalloc.restype = ctypes.c_int
    L.pa_copy_blocks.argtypes = [vp, vp, ctypes.POINTER(CacheDesc), vp, i32, vp, vp]
    L.pa_copy_blocks.restype = ctypes.c_int
    i64 = ctypes.c_int64
    L.pa_bm_create.argtypes = [i32, i32]
    L.pa_bm_create.restype = vp
    L.pa_bm_destroy.argtypes = [vp]
    L.pa_bm_destroy.restype = None
    L.pa_bm_num_free.argtypes = [vp]
    L.pa_bm_num_free.restype = i32
    L.pa_bm_append.argtypes = [vp, i64, i32, vp, vp, i32]
    L.pa_bm_append.restype = i32
    L.pa_bm_append_tokens.argtypes = [vp, i64, vp, i32, vp, vp, i32, vp]
    L.pa_bm_append_tokens.restype = i32
    L.pa_bm_cached_prefix.argtypes = [vp, vp, i32]
    L.pa_bm_cached_prefix.restype = i32
    L.pa_bm_fork.argtypes = [vp, i64, i64]
    L.pa_bm_fork.restype = i32
    L.pa_bm_free.argtypes = [vp, i64]
    L.pa_bm_free.restype = i32
    L.pa_bm_block_table.argtypes = [vp, i64, vp, i32]
    L.pa_bm_block_table.restype = i32
    L.pa_bm_num_tokens.argtypes = [vp, i64]
    L.pa_bm_num_tokens.restype = i64
    L.pa_bm_refcount.argtypes = [vp, i32]
    L.pa_bm_refcount.restype = i32
    L.pa_check_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.pa_check_error.restype = ctypes.c_int
    L.pa_workspace_init.argtypes = [vp, vp]
    L.pa_workspace_init.restype = ctypes.c_int
    L.pa_last_error_string.argtypes = []
    L.pa_last_error_string.restype = ctypes.c_char_p
    L.pa_version.argtypes = []
    L.pa_version.restype = ctypes.c_char_p
    L.pa_set_kernel_timing_events.argtypes = [vp, vp]
    L.pa_set_kernel_timing_events.restype = None
    L.pa_set_prefill_timing_events.argtypes = [vp, vp]
    L.pa_set_prefill_timing_events.restype = None
    L.pa_set_kernel_span_buffer.argtypes = [vp]
    L.pa_set_kernel_span_buffer.restype = None
    L.pa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.pa_set_wait_limit_ns.restype = None
    L.pa_test_skip_one_copy.argtypes = [i32]
    L.pa_test_skip_one_copy.restype = None
    L.pa_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    L.pa_selftest_wait_timeout.restype = ctypes.c_int
    _LIB = L
    return L


def check(status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, load().pa_last_error_string().decode())
