"""The allocation-free decode entry point (bsp_decode_run_static).

Some callers cannot allocate device memory where they run attention: a
serving engine whose KV-cache manager reserved nearly all of HBM for its own
pool and allows no further allocation while it serves, or a plugin that its
host hands only input and output tensors. bsp_decode_run_static keeps the
run's scratch in a fixed array inside the library instead.

These tests drive it through the C ABI. On two calls in a row with different
plans (so that what the first call leaves in the shared array could leak into
the second), each call must give bit for bit what the regular entry point
(bsp_decode_run with the caller's workspace) gives on the same plan with the
same cp.async gather (num_pages = 0), match the oracle at the bf16 bounds of
the other parity tests, and leave the device's free memory unchanged. This
file is collected last, and passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare, lib, oracle_full, to_dev

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_static_workspace_matches_caller_workspace_twice():
    bsp = lib()
    N = bsp._native
    lb = N.load()
    calls = [
        (61, [4000, 17, 900, 0, 2500, 64, 7000], 64),   # split outputs: partial states are used
        (62, [300, 5000, 33], 40),                        # a different plan over the same array
    ]
    for i, (seed, kv, C) in enumerate(calls):
        b = workloads.paged_batch(seed, np.ones(len(kv), int), kv, 32, 8, 128, 16, "bf16", extra_pages=3)
        q, k, v, idx = to_dev(b)
        pa = bsp.PagedAttention("decode", 32, 8, 128, 16, False, torch.bfloat16, max_batch=b.batch, num_ctas=C)
        pa.plan(b.kv_indptr, b.last_page_len)   # staging image (pinned) + the copy into pa.workspace
        torch.cuda.synchronize()
        assert pa.info.workspace_bytes <= N.BSP_STATIC_WORKSPACE_BYTES
        if seed == 61:
            assert pa.info.num_merges > 0
        ref_o, ref_l = torch.empty_like(q), torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        out, lse = torch.empty_like(q), torch.empty_like(ref_l)
        N.check(lb.bsp_decode_run(ctypes.byref(pa.info), _p(q), _p(k), _p(v), _p(idx), 0,
                                  ctypes.c_float(b.sm_scale), _p(ref_o), _p(ref_l), _p(pa.workspace), _stream()))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        N.check(lb.bsp_decode_run_static(ctypes.byref(pa.info), ctypes.c_void_p(pa.staging.data_ptr()), _p(q),
                                         _p(k), _p(v), _p(idx), ctypes.c_float(b.sm_scale), _p(out), _p(lse),
                                         _stream()))
        torch.cuda.synchronize()
        if i > 0:  # the first call on the device may load the library's module
            assert torch.cuda.mem_get_info()[0] == free0, "the static entry point changed the free device memory"
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        O, L = oracle_full(b)
        compare(out, lse, O, L, "bf16")


def test_static_workspace_rejects_bad_plans():
    bsp = lib()
    N = bsp._native
    lb = N.load()
    b = workloads.paged_batch(63, [1, 1], [10, 20], 32, 8, 128, 16, "bf16")
    q, k, v, idx = to_dev(b)
    out = torch.empty_like(q)

    def call(info, staging):
        return lb.bsp_decode_run_static(ctypes.byref(info), staging.ctypes.data_as(ctypes.c_void_p), _p(q), _p(k),
                                        _p(v), _p(idx), ctypes.c_float(b.sm_scale), _p(out), None, _stream())

    def host_plan(capacity):
        problem = bsp.make_problem(bsp.BSP_MODE_DECODE, 32, 8, 128, 16, False, torch.bfloat16)
        staging = np.zeros(lb.bsp_host_staging_size(ctypes.byref(problem), ctypes.byref(capacity)), np.uint8)
        kv = np.ascontiguousarray(b.kv_indptr, np.int32)
        lp = np.ascontiguousarray(b.last_page_len, np.int32)
        info = N.PlanInfo()
        N.check(lb.bsp_plan(ctypes.byref(problem), ctypes.byref(capacity), b.batch, None,
                            kv.ctypes.data_as(ctypes.c_void_p), lp.ctypes.data_as(ctypes.c_void_p), 2, 1,
                            staging.ctypes.data_as(ctypes.c_void_p), None, 0, None, ctypes.byref(info)))
        return info, staging

    # 40000 partial slots: far beyond the static array
    info, staging = host_plan(N.Capacity(2, 20000, 2))
    assert info.workspace_bytes > N.BSP_STATIC_WORKSPACE_BYTES
    assert call(info, staging) == N.BSP_ERR_CAPACITY
    assert b"BSP_STATIC_WORKSPACE_BYTES" in lb.bsp_last_error()
    # counts or offsets that do not fit the plan's own layout
    info, staging = host_plan(N.Capacity(2, 8, 2))
    for field, value in (("num_items", info.cap_items + 1), ("off_merges", info.off_merges + 64)):
        bad = N.PlanInfo()
        ctypes.pointer(bad)[0] = info
        setattr(bad, field, value)
        assert call(bad, staging) == N.BSP_ERR_INVALID_ARG
    torch.cuda.synchronize()
