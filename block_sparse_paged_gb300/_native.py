"""ctypes view of libbsp.so (the C ABI declared in include/bsp.h).

Argument marshalling only. If the library is missing this module raises: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbsp.so")

BSP_OK = 0
BSP_ERR_INVALID_ARG = -1
BSP_ERR_CAPACITY = -2
BSP_ERR_CUDA = -3
BSP_ERR_UNSUPPORTED = -4
BSP_ERR_DEVICE_CHECK = -5

BSP_DTYPE_BF16 = 0
BSP_DTYPE_F32 = 1
BSP_SCHEDULE_LPT = 0
BSP_SCHEDULE_EQUAL_SHARES = 1
BSP_MODE_DECODE = 0
BSP_MODE_PREFILL = 1
BSP_STATIC_WORKSPACE_BYTES = 8 << 20

_ERR_NAMES = {BSP_ERR_INVALID_ARG: "INVALID_ARG", BSP_ERR_CAPACITY: "CAPACITY", BSP_ERR_CUDA: "CUDA",
              BSP_ERR_UNSUPPORTED: "UNSUPPORTED", BSP_ERR_DEVICE_CHECK: "DEVICE_CHECK"}

EXPORTED = ["bsp_default_num_ctas", "bsp_workspace_size", "bsp_host_staging_size", "bsp_plan",
            "bsp_decode_run", "bsp_decode_run_fp8", "bsp_prefill_run", "bsp_run_attention", "bsp_run_merge_partials",
            "bsp_merge_state", "bsp_decode_run_static", "bsp_check_device_error", "bsp_check_bounded_wait",
            "bsp_last_error", "bsp_version"]


class Problem(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("window_left", ctypes.c_int32), ("logits_soft_cap", ctypes.c_float),
                ("sink", ctypes.c_void_p)]


class Capacity(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("max_qo_tokens", ctypes.c_int64),
                ("chunks_per_cta", ctypes.c_int32), ("max_gather_pages", ctypes.c_int32),
                ("schedule", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("problem", Problem), ("capacity", Capacity), ("batch", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("group", ctypes.c_int32), ("chunk_len", ctypes.c_int32),
                ("total_work", ctypes.c_int64), ("alpha", ctypes.c_int64), ("beta", ctypes.c_int64),
                ("num_items", ctypes.c_int32), ("num_merges", ctypes.c_int32), ("num_partials", ctypes.c_int32),
                ("cap_items", ctypes.c_int32), ("cap_merges", ctypes.c_int32), ("cap_partials", ctypes.c_int32),
                ("off_header", ctypes.c_uint64), ("off_queue_indptr", ctypes.c_uint64),
                ("off_items", ctypes.c_uint64), ("off_merges", ctypes.c_uint64), ("off_status", ctypes.c_uint64),
                ("off_partial_lse", ctypes.c_uint64), ("off_partial_o", ctypes.c_uint64),
                ("metadata_bytes", ctypes.c_uint64), ("workspace_bytes", ctypes.c_uint64),
                ("valid", ctypes.c_int32), ("num_qo_tokens", ctypes.c_int32),
                ("num_table_pages", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("off_gather", ctypes.c_uint64), ("gather_pool_bytes", ctypes.c_uint64)]


# numpy views of the plan's staging image (bsp_work_item, bsp_merge_entry)
WORK_ITEM_DTYPE = np.dtype([("b", "<i4"), ("tile", "<i4"), ("kv_head", "<i4"), ("kv_start", "<i4"),
                            ("kv_end", "<i4"), ("slot", "<i4"), ("q_tok0", "<i4"), ("n_pos", "<i4"),
                            ("qo_len", "<i4"), ("kv_len", "<i4"), ("page_base", "<i4"), ("pos0", "<i4"),
                            ("merge", "<i4"), ("reserved", "<i4", (3,))])
MERGE_ENTRY_DTYPE = np.dtype([("b", "<i4"), ("tile", "<i4"), ("kv_head", "<i4"), ("slot_begin", "<i4"),
                              ("n_slots", "<i4"), ("q_tok0", "<i4"), ("n_pos", "<i4"), ("arrived", "<i4")])
assert WORK_ITEM_DTYPE.itemsize == 64 and MERGE_ENTRY_DTYPE.itemsize == 32


class BspError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"bsp error {_ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load():
    """Load libbsp.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m block_sparse_paged_gb300.build` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    P, C, PI = ctypes.POINTER(Problem), ctypes.POINTER(Capacity), ctypes.POINTER(PlanInfo)
    sig = {
        "bsp_default_num_ctas": ([i32, i32, ctypes.POINTER(i32)], ctypes.c_int),
        "bsp_workspace_size": ([P, C], ctypes.c_size_t),
        "bsp_host_staging_size": ([P, C], ctypes.c_size_t),
        "bsp_plan": ([P, C, i32, vp, vp, vp, i64, i64, vp, vp, ctypes.c_size_t, vp, PI], ctypes.c_int),
        "bsp_decode_run": ([PI, vp, vp, vp, vp, i64, f32, vp, vp, vp, vp], ctypes.c_int),
        "bsp_decode_run_fp8": ([PI, vp, vp, vp, vp, i64, f32, f32, f32, vp, vp, vp, vp], ctypes.c_int),
        "bsp_prefill_run": ([PI, vp, vp, vp, vp, i64, f32, vp, vp, vp, vp], ctypes.c_int),
        "bsp_run_attention": ([PI, vp, vp, vp, vp, i64, f32, vp, vp, vp, vp], ctypes.c_int),
        "bsp_run_merge_partials": ([PI, vp, vp, vp, vp], ctypes.c_int),
        "bsp_merge_state": ([vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp], ctypes.c_int),
        "bsp_decode_run_static": ([PI, vp, vp, vp, vp, vp, f32, vp, vp, vp], ctypes.c_int),
        "bsp_check_device_error": ([PI, vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "bsp_check_bounded_wait": ([i64, vp, vp], ctypes.c_int),
        "bsp_last_error": ([], ctypes.c_char_p),
        "bsp_version": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def check(rc: int) -> None:
    if rc != BSP_OK:
        raise BspError(rc, load().bsp_last_error().decode())
