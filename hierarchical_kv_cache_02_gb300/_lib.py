"""ctypes declarations of the C ABI in include/hisparse.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

HS_OK, HS_ERR_CONFIG, HS_ERR_ALLOC_HOST, HS_ERR_ALLOC_DEV, HS_ERR_ARG, HS_ERR_CUDA, HS_ERR_DEVICE_FLAG = (
    0, -1, -2, -3, -4, -5, -6)
HS_ERR_SCRATCH = -7
STATUS_NAMES = {0: "HS_OK", -1: "HS_ERR_CONFIG", -2: "HS_ERR_ALLOC_HOST", -3: "HS_ERR_ALLOC_DEV",
                -4: "HS_ERR_ARG", -5: "HS_ERR_CUDA", -6: "HS_ERR_DEVICE_FLAG", -7: "HS_ERR_SCRATCH"}
POLICY_LRU, POLICY_FIFO, POLICY_RANDOM, POLICY_SWAP_VANILLA = 0, 1, 2, 3
LAYOUT_MLA, LAYOUT_GQA = 0, 1
DEVERR_RANGE, DEVERR_DUP, DEVERR_CLOCK, DEVERR_APPEND, DEVERR_LOC, DEVERR_TIMEOUT = 1, 2, 4, 8, 16, 32
DEVERR_PAGE, DEVERR_SLOTS = 64, 128
STALL_ATTN, STALL_RESOLVE, STALL_FETCH = 1, 2, 4  # hs_debug_stall_next (test hook for the bounded waits)

# every entry point include/hisparse.h declares
EXPORTS = ("hs_record_bytes", "hs_pool_create", "hs_pool_destroy", "hs_pool_reset", "hs_prefill_write",
           "hs_append_writethrough", "hs_resolve", "hs_sparse_attn", "hs_stats", "hs_read_state",
           "hs_read_buffer", "hs_read_history", "hs_sparse_attn_noalloc", "hs_append_resolve",
           "hs_resolve_range", "hs_sparse_attn_range", "hs_reserve", "hs_release", "hs_host_usage",
           "hs_device_usage", "hs_debug_stall_next")


class hs_config(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("capacity", ctypes.c_int64),
        ("shared_prefix", ctypes.c_int64),
        ("layout", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("buffer_slots", ctypes.c_int32),
        ("policy", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("io_chunk_bytes", ctypes.c_int32),
        ("log_steps", ctypes.c_int32),
        ("fetch_in_attention", ctypes.c_int32),
        ("host_page_tokens", ctypes.c_int32),
        ("host_on_demand", ctypes.c_int32),
        ("buffer_page_slots", ctypes.c_int32),
        ("device_pool_slots", ctypes.c_int64),
        ("host_to_device_ratio", ctypes.c_double),
        ("early_fetch", ctypes.c_int32),
    ]


class hs_totals(ctypes.Structure):
    _fields_ = [
        ("hits", ctypes.c_uint64),
        ("misses", ctypes.c_uint64),
        ("appends", ctypes.c_uint64),
        ("host_bytes", ctypes.c_uint64),
        ("error_bits", ctypes.c_uint32),
        ("resolves", ctypes.c_uint32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libhisparse.so.  Raises if it has not been built: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(f"{path} is missing: build it with hierarchical_kv_cache_02_gb300.build."
                                  "build_library() (the CUDA library is required; there is no CPU path)")
            _build.build_library()
        lib = ctypes.CDLL(path)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        sig = {
            "hs_record_bytes": (I64, [P]),
            "hs_pool_create": (I, [P, I, P]),
            "hs_pool_destroy": (I, [P]),
            "hs_pool_reset": (I, [P, P]),
            "hs_prefill_write": (I, [P, I, I, I64, I64, P, P]),
            "hs_append_writethrough": (I, [P, I, P, P, P]),
            "hs_resolve": (I, [P, I, P, P, P]),
            "hs_sparse_attn": (I, [P, I, P, P, P, I64, F, P, P]),
            "hs_stats": (I, [P, P, P, P, P, I]),
            "hs_read_state": (I, [P, I, P, P, P]),
            "hs_read_buffer": (I, [P, I, I, P]),
            "hs_read_history": (I, [P, I, I, I64, I64, P]),
            "hs_sparse_attn_noalloc": (I, [P, P, P, P, I64, F, P, P]),
            "hs_append_resolve": (I, [P, I, P, P, P, P, P]),
            "hs_resolve_range": (I, [P, I, I, I, P, P, P, P, P]),
            "hs_sparse_attn_range": (I, [P, I, I, I, P, P, F, P, P]),
            "hs_reserve": (I, [P, I, I, I64]),
            "hs_release": (I, [P, I]),
            "hs_host_usage": (I, [P, P, P, P]),
            "hs_device_usage": (I, [P, P, P, P]),
            "hs_debug_stall_next": (I, [P, I]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return _lib
