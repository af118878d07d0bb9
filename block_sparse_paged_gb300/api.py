"""Thin Python binding of the C ABI: torch tensors in, pointers to libbsp.so out.

Every step of the path runs in the library's kernels; this module only checks
shapes, dtypes and devices and passes pointers, sizes and the current stream.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from . import _native as N

_DTYPES = {torch.bfloat16: N.BSP_DTYPE_BF16, torch.float32: N.BSP_DTYPE_F32}


def _i32_host(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _stream_handle(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, device=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return ctypes.c_void_p(t.data_ptr())


def default_num_ctas(mode: int, device: int | None = None) -> int:
    dev = torch.cuda.current_device() if device is None else device
    out = ctypes.c_int32()
    N.check(N.load().bsp_default_num_ctas(mode, dev, ctypes.byref(out)))
    return int(out.value)


def make_problem(mode: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 causal: bool, dtype, window_left: int = -1, logits_soft_cap: float = 0.0) -> N.Problem:
    return N.Problem(mode, num_qo_heads, num_kv_heads, head_dim, page_size, int(bool(causal)), _DTYPES[dtype],
                     int(window_left), float(logits_soft_cap))


def plan_host(problem: N.Problem, capacity: N.Capacity, kv_indptr, last_page_len, qo_indptr=None,
              alpha: int = 2, beta: int = 1):
    """Plan on the host only (no device, nothing copied): returns
    (info, queue_indptr, items, merges) read back from the staging image."""
    lib = N.load()
    nbytes = lib.bsp_host_staging_size(ctypes.byref(problem), ctypes.byref(capacity))
    if nbytes == 0:
        N.check(N.BSP_ERR_INVALID_ARG)
    staging = np.zeros(nbytes, np.uint8)
    kv = _i32_host(kv_indptr)
    lp = _i32_host(last_page_len)
    qo = None if qo_indptr is None else _i32_host(qo_indptr)
    info = N.PlanInfo()
    N.check(lib.bsp_plan(ctypes.byref(problem), ctypes.byref(capacity), len(kv) - 1,
                         None if qo is None else _ptr(qo), _ptr(kv), _ptr(lp), alpha, beta,
                         _ptr(staging), None, 0, None, ctypes.byref(info)))
    return (info,) + read_plan(info, staging)


def read_plan(info: N.PlanInfo, staging: np.ndarray):
    """(queue_indptr [C+1], items, merges) from a staging image."""
    C = info.capacity.num_ctas
    q = staging[info.off_queue_indptr: info.off_queue_indptr + 4 * (C + 1)].view(np.int32).copy()
    items = staging[info.off_items: info.off_items + 64 * info.num_items].view(N.WORK_ITEM_DTYPE).copy()
    merges = staging[info.off_merges: info.off_merges + 32 * info.num_merges].view(N.MERGE_ENTRY_DTYPE).copy()
    return q, items, merges


class PagedAttention:
    """Workspace, plan and runs of block-sparse paged attention for one problem.

    mode: "decode" (one query per request, the g heads of a kv head fused into
    one tile) or "prefill" (ragged queries, 256-row tiles, tensor cores).
    max_gather_pages (prefill): pages of a K / V copy region in the workspace;
    prefills whose pages are under 8 tokens (or not a power of two) and whose
    page table fits it are gathered into it first and then read by TMA.
    schedule: "lpt" (the pages' plan) or "equal" (equal contiguous shares of
    the concatenated KV ranges per CTA, for batches of few, equal tiles).
    The workspace and pinned staging buffer are allocated once, for the
    given bounds; plan() may then be called once per step and run() once per
    layer, and run() can be captured in a CUDA graph.
    """

    def __init__(self, mode: str, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 causal: bool = False, dtype=torch.bfloat16, max_batch: int = 256,
                 max_qo_tokens: int | None = None, num_ctas: int | None = None, device=None,
                 window_left: int = -1, logits_soft_cap: float = 0.0, chunks_per_cta: int = 1,
                 max_gather_pages: int = 0, schedule: str = "lpt"):
        self.lib = N.load()
        if mode not in ("decode", "prefill"):
            raise ValueError("mode must be 'decode' or 'prefill'")
        self.mode = N.BSP_MODE_DECODE if mode == "decode" else N.BSP_MODE_PREFILL
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.dtype = dtype
        self.problem = make_problem(self.mode, num_qo_heads, num_kv_heads, head_dim, page_size, causal, dtype,
                                    window_left, logits_soft_cap)
        if num_ctas is None:
            num_ctas = default_num_ctas(self.mode, self.device.index)
        if max_qo_tokens is None:
            max_qo_tokens = max_batch if mode == "decode" else 65536
        if schedule not in ("lpt", "equal"):
            raise ValueError("schedule must be 'lpt' or 'equal'")
        sched = N.BSP_SCHEDULE_LPT if schedule == "lpt" else N.BSP_SCHEDULE_EQUAL_SHARES
        self.capacity = N.Capacity(max_batch, num_ctas, max_qo_tokens, chunks_per_cta, max_gather_pages, sched)
        ws_bytes = self.lib.bsp_workspace_size(ctypes.byref(self.problem), ctypes.byref(self.capacity))
        st_bytes = self.lib.bsp_host_staging_size(ctypes.byref(self.problem), ctypes.byref(self.capacity))
        if ws_bytes == 0 or st_bytes == 0:
            N.check(N.BSP_ERR_INVALID_ARG)
        self.workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=self.device)
        self.staging = torch.zeros(st_bytes, dtype=torch.uint8, pin_memory=True)
        self._copied = None  # event after the last plan copy
        self.info = None

    # ---- plan ---------------------------------------------------------------
    # Default per-position cost alpha of the LPT plan (cost of a work item =
    # alpha * query positions + beta * KV tokens). The pages' constants are
    # alpha = 2, beta = 1; a decode work item (one position) costs more than 2
    # tokens of KV on this GPU: about 64 (its setup and epilogue, measured as the
    # alpha that balanced a batch of short requests best: 59.0 -> 55.5 us).
    DEFAULT_ALPHA = {N.BSP_MODE_DECODE: 64, N.BSP_MODE_PREFILL: 2}

    def plan(self, kv_indptr, last_page_len, qo_indptr=None, alpha: int | None = None, beta: int = 1, stream=None):
        """Host plan from the request lengths; its copy is queued on `stream`.
        alpha defaults to DEFAULT_ALPHA[mode]."""
        if alpha is None:
            alpha = self.DEFAULT_ALPHA[self.mode]
        if self._copied is not None:
            self._copied.synchronize()  # the staging buffer is still the source of the previous copy
        kv = _i32_host(kv_indptr)
        lp = _i32_host(last_page_len)
        qo = None if qo_indptr is None else _i32_host(qo_indptr)
        info = N.PlanInfo()
        with torch.cuda.device(self.device):
            s = _stream_handle(stream)
            N.check(self.lib.bsp_plan(ctypes.byref(self.problem), ctypes.byref(self.capacity), len(kv) - 1,
                                      None if qo is None else _ptr(qo), _ptr(kv), _ptr(lp), alpha, beta,
                                      ctypes.c_void_p(self.staging.data_ptr()),
                                      ctypes.c_void_p(self.workspace.data_ptr()), self.workspace.numel(), s,
                                      ctypes.byref(info)))
            ev = torch.cuda.Event()
            ev.record(stream if stream is not None else torch.cuda.current_stream())
            self._copied = ev
        self.info = info
        return info

    def plan_arrays(self):
        """(queue_indptr, items, merges) of the current plan (host copy)."""
        return read_plan(self.info, self.staging.numpy())

    # ---- run ----------------------------------------------------------------
    def run(self, q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, kv_indices: torch.Tensor,
            sm_scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
            stream=None, return_lse: bool = True, k_scale: float = 1.0, v_scale: float = 1.0,
            sink: torch.Tensor | None = None):
        """Attention of the planned batch. k_pages / v_pages are in the
        problem's dtype, or, for bf16 decode, torch.float8_e4m3fn pools read as
        k_scale * k_pages and v_scale * v_pages (one scale per pool). sink:
        float32 [H_qo] on the device, one extra softmax logit per query head
        without a value row (the attention-sink variant), or None."""
        if self.info is None:
            raise RuntimeError("plan() must be called before run()")
        P = self.problem
        D = P.head_dim
        if q.dim() != 3 or q.shape[1] != P.num_qo_heads or q.shape[2] != D:
            raise ValueError(f"q must be [n_tokens, {P.num_qo_heads}, {D}]")
        if k_pages.dim() != 4 or k_pages.shape[1:] != (P.page_size, P.num_kv_heads, D) or v_pages.shape != k_pages.shape:
            raise ValueError(f"k_pages / v_pages must be [num_pages, {P.page_size}, {P.num_kv_heads}, {D}]")
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        dev = self.device
        fp8 = k_pages.dtype == torch.float8_e4m3fn
        if fp8 and (self.mode != N.BSP_MODE_DECODE or self.dtype != torch.bfloat16):
            raise ValueError("e4m3 KV pools are read by the bf16 decode run only")
        kv_dt = torch.float8_e4m3fn if fp8 else self.dtype
        if not fp8 and (k_scale != 1.0 or v_scale != 1.0):
            raise ValueError("k_scale / v_scale apply to e4m3 KV pools only")
        args = [ctypes.byref(self.info), _dev(q, "q", self.dtype, dev), _dev(k_pages, "k_pages", kv_dt, dev),
                _dev(v_pages, "v_pages", kv_dt, dev), _dev(kv_indices, "kv_indices", torch.int32, dev)
                if kv_indices.numel() else None]
        tail = [ctypes.c_float(sm_scale), _dev(out, "out", self.dtype, dev),
                None if lse is None else _dev(lse, "lse", torch.float32, dev),
                ctypes.c_void_p(self.workspace.data_ptr())]
        self._set_sink(sink)
        with torch.cuda.device(dev):
            s = _stream_handle(stream)
            if fp8:
                N.check(self.lib.bsp_decode_run_fp8(*args, k_pages.shape[0], tail[0], ctypes.c_float(k_scale),
                                                    ctypes.c_float(v_scale), *tail[1:], s))
            elif self.mode == N.BSP_MODE_DECODE:
                N.check(self.lib.bsp_decode_run(*args, k_pages.shape[0], *tail, s))
            else:
                N.check(self.lib.bsp_prefill_run(*args, k_pages.shape[0], *tail, s))
        return (out, lse) if return_lse else out

    def _set_sink(self, sink):
        if sink is None:
            self.info.problem.sink = None
            return
        if sink.dim() != 1 or sink.shape[0] != self.problem.num_qo_heads:
            raise ValueError(f"sink must be [{self.problem.num_qo_heads}]")
        self.info.problem.sink = _dev(sink, "sink", torch.float32, self.device).value
        self._sink_ref = sink  # the kernel reads it during the run

    def run_stages(self, q, k_pages, v_pages, kv_indices, sm_scale, out, lse, stream=None, events=None):
        """The run as its launches on `stream`: the attention kernel, then for
        prefill the merge of partials (decode merges inside its kernel);
        `events` = (e0, e1, e2) are recorded before, between and after them when
        given. out and lse must be preallocated."""
        dev = self.device
        with torch.cuda.device(dev):
            st = stream if stream is not None else torch.cuda.current_stream()
            s = ctypes.c_void_p(st.cuda_stream)
            ws = ctypes.c_void_p(self.workspace.data_ptr())
            o_p = _dev(out, "out", self.dtype, dev)
            l_p = None if lse is None else _dev(lse, "lse", torch.float32, dev)
            self._set_sink(None)
            if events:
                events[0].record(st)
            N.check(self.lib.bsp_run_attention(ctypes.byref(self.info), _dev(q, "q", self.dtype, dev),
                                               _dev(k_pages, "k_pages", self.dtype, dev),
                                               _dev(v_pages, "v_pages", self.dtype, dev),
                                               _dev(kv_indices, "kv_indices", torch.int32, dev), k_pages.shape[0],
                                               ctypes.c_float(sm_scale), o_p, l_p, ws, s))
            if events:
                events[1].record(st)
            if self.mode == N.BSP_MODE_PREFILL:  # decode merges split outputs inside its kernel
                N.check(self.lib.bsp_run_merge_partials(ctypes.byref(self.info), o_p, l_p, ws, s))
            if events:
                events[2].record(st)
        return out, lse

    def check_device_error(self, stream=None) -> int:
        word = ctypes.c_int32()
        with torch.cuda.device(self.device):
            N.check(self.lib.bsp_check_device_error(ctypes.byref(self.info), ctypes.c_void_p(self.workspace.data_ptr()),
                                                    _stream_handle(stream), ctypes.byref(word)))
        return int(word.value)


def merge_state(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor, lse_b: torch.Tensor,
                out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None, stream=None):
    """Merge two sets of attention states O [n, H, D], LSE [n, H] (float32)."""
    if o_a.shape != o_b.shape or o_a.dim() != 3 or lse_a.shape != o_a.shape[:2] or lse_b.shape != lse_a.shape:
        raise ValueError("o_a, o_b must be [n, H, D] and lse_a, lse_b [n, H]")
    dt = o_a.dtype
    if dt not in _DTYPES:
        raise ValueError("dtype must be bfloat16 or float32")
    if out is None:
        out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    n, H, D = o_a.shape
    lib = N.load()
    with torch.cuda.device(o_a.device):
        N.check(lib.bsp_merge_state(_dev(o_a, "o_a", dt), _dev(lse_a, "lse_a", torch.float32), _dev(o_b, "o_b", dt),
                                    _dev(lse_b, "lse_b", torch.float32), _dev(out, "out", dt),
                                    _dev(lse_out, "lse_out", torch.float32), n, H, D, _DTYPES[dt],
                                    _stream_handle(stream)))
    return out, lse_out
