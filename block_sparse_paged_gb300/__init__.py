"""Block-sparse paged attention for GB300 (sm_103a).

The hot path is the C-ABI library libbsp.so (include/bsp.h): a host planner
and hand-written CUDA kernels for paged decode, ragged prefill and the exact
merge of attention states. This package is its thin Python binding. The
library is loaded on first use (so that ``block_sparse_paged_gb300.build`` can
rebuild it first); every entry point raises if it has not been built.
"""
from . import _native
from ._native import (BSP_DTYPE_BF16, BSP_DTYPE_F32, BSP_MODE_DECODE, BSP_MODE_PREFILL, BspError, Capacity,
                      PlanInfo, Problem)
from .api import PagedAttention, default_num_ctas, make_problem, merge_state, plan_host, read_plan


__all__ = ["PagedAttention", "merge_state", "plan_host", "read_plan", "default_num_ctas", "make_problem",
           "Problem", "Capacity", "PlanInfo", "BspError", "BSP_DTYPE_BF16", "BSP_DTYPE_F32",
           "BSP_MODE_DECODE", "BSP_MODE_PREFILL"]
