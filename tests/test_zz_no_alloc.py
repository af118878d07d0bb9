"""The allocation-free decode entry point (bsp_decode_run_static).

It exists for callers that may not call cudaMalloc where they run attention:
a serving framework that gave all device memory to its own pool and forbids
allocation while serving, or code running inside a global-mode stream
capture. The test drives it through the C ABI with a host-only plan and
checks it against the regular entry point (bsp_decode_run with a workspace
the caller allocated), at the tolerances of the other parity tests, on two
calls in a row with different plans, so that what the first call leaves in
the shared array cannot leak into the second. This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import TOL, lib, run_batch, to_dev

pytestmark = pytest.mark.gpu


def host_plan(N, problem, capacity, batch):
    """A host-only plan (no workspace) and the staging image it was written to."""
    lb = N.load()
    staging = np.zeros(lb.bsp_host_staging_size(ctypes.byref(problem), ctypes.byref(capacity)), np.uint8)
    kv = np.ascontiguousarray(batch.kv_indptr, np.int32)
    lp = np.ascontiguousarray(batch.last_page_len, np.int32)
    info = N.PlanInfo()
    N.check(lb.bsp_plan(ctypes.byref(problem), ctypes.byref(capacity), batch.batch, None,
                        kv.ctypes.data_as(ctypes.c_void_p), lp.ctypes.data_as(ctypes.c_void_p), 2, 1,
                        staging.ctypes.data_as(ctypes.c_void_p), None, 0, None, ctypes.byref(info)))
    return info, staging


def static_run(N, info, staging, batch):
    q, k, v, idx = to_dev(batch)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    N.check(N.load().bsp_decode_run_static(ctypes.byref(info), staging.ctypes.data_as(ctypes.c_void_p), ptr(q),
                                           ptr(k), ptr(v), ptr(idx), ctypes.c_float(batch.sm_scale), ptr(out),
                                           ptr(lse), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    return out, lse


def test_static_workspace_matches_caller_workspace_twice():
    bsp = lib()
    N = bsp._native
    calls = [
        (61, [4000, 17, 900, 0, 2500, 64, 7000], 64),   # split outputs: partial states are used
        (62, [300, 5000, 33], 40),                        # a different plan over the same array
    ]
    for seed, kv, C in calls:
        b = workloads.paged_batch(seed, np.ones(len(kv), int), kv, 32, 8, 128, 16, "bf16", extra_pages=3)
        ref_out, ref_lse, pa = run_batch(bsp, b, num_ctas=C)
        info, staging = host_plan(N, pa.problem, pa.capacity, b)
        assert info.workspace_bytes <= N.BSP_STATIC_WORKSPACE_BYTES
        if seed == 61:
            assert info.num_merges > 0
        out, lse = static_run(N, info, staging, b)
        tol_o, tol_l = TOL["bf16"]
        empty = torch.isneginf(ref_lse)
        assert torch.equal(torch.isneginf(lse), empty)
        assert (out.float() - ref_out.float()).abs().max().item() <= tol_o
        assert (lse[~empty] - ref_lse[~empty]).abs().max().item() <= tol_l


def test_static_workspace_rejects_oversized_plans():
    bsp = lib()
    N = bsp._native
    b = workloads.paged_batch(63, [1, 1], [10, 20], 32, 8, 128, 16, "bf16")
    problem = bsp.make_problem(bsp.BSP_MODE_DECODE, 32, 8, 128, 16, False, torch.bfloat16)
    capacity = N.Capacity(2, 20000, 2)   # 40000 partial slots: far beyond the static array
    info, staging = host_plan(N, problem, capacity, b)
    assert info.workspace_bytes > N.BSP_STATIC_WORKSPACE_BYTES
    q, k, v, idx = to_dev(b)
    out = torch.empty_like(q)
    rc = N.load().bsp_decode_run_static(ctypes.byref(info), staging.ctypes.data_as(ctypes.c_void_p),
                                        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(idx.data_ptr()),
                                        ctypes.c_float(b.sm_scale), ctypes.c_void_p(out.data_ptr()), None,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == N.BSP_ERR_CAPACITY
    assert b"BSP_STATIC_WORKSPACE_BYTES" in N.load().bsp_last_error()
