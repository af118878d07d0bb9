#!/usr/bin/env python
"""Benchmark of the block-sparse paged attention path on GB300.

Step = plan() on the host + the attention kernel + the merge of split
outputs, over the Llama-3-8B-shaped batched paged decode (64 requests, KV
lengths U{512..8192}, page size 16, pages permuted over the pool, 32 qo / 8 kv
heads, head_dim 128, bf16), inputs resident in HBM. value = algorithmic bytes
of the step (KV + Q + O + LSE + page table) / step time, in GB/s.

Also reported: the attention kernel's roofline against the measured HBM
copy bandwidth, the same metric end to end through the public API with host
buffers (host->device copies of every input and device->host copy of O and
LSE inside the timed region), the oracle on the host cores, the SM clocks
sampled during the timed region, and secondary workloads (page-size-1 decode
permuted vs contiguous, ragged causal prefill TFLOP/s, shared-prefix decode).

Multi-GPU: one process per GPU under torch.distributed.run; every rank runs
its own replica of the workload (the path shards by request, no data-path
collective), timing is max over ranks and value sums all ranks' bytes.
`--impl reference` times the oracle (the plain fp64 CPU implementation) as
the reference arm, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-KV decode GB/s & ragged prefill TFLOPS, % of GB300 roofline (1 GPU)"
WORKLOAD = "batched_decode_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# sources whose digest keys the committed ncu traffic figures (profiles/traffic.json)
DECODE_SOURCES = ("decode.cu", "tmap.cpp", "device_common.cuh", "sm100.cuh", "bsp_internal.h")
PREFILL_SOURCES = ("prefill.cu", "tmap.cpp", "device_common.cuh", "sm100.cuh", "bsp_internal.h")


# ---------------------------------------------------------------------------
# distributed plumbing (timing only; the data path has no collective)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# measured peaks, clocks, profile summaries
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        try:
            rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
            os.unlink(self.path)
        except OSError:
            return None
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(pw) if pw else None}


def clocks_while(run, seconds: float, gpu_index: int):
    """SM clocks (ClockSampler) while run() is called back to back for about
    `seconds`: the clock a kernel holds under its own sustained load."""
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_index).start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            run()
        torch.cuda.synchronize()
    return sampler.stop()


def kernel_digest(*names) -> str:
    """Digest of the kernel sources with comments and whitespace removed (the
    sources hold no comment markers inside string literals), so that an edit of
    comments alone keeps a capture valid."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_paged_gb300", "csrc", n), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profile_traffic(key: str, digest: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[key]
        if e.get("source_digest") == digest:
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def esize(batch) -> int:
    return 2 if batch.dtype == "bf16" else 4


def decode_bytes(batch) -> int:
    """Bytes a decode step must move at least once: K and V of every visible
    token of every kv head, Q, O, LSE and the page table."""
    e = esize(batch)
    kv = int(batch.kv_lens.sum()) * batch.num_kv_heads * batch.head_dim * e * 2
    n_tok = int(batch.qo_indptr[-1])
    qo = 2 * n_tok * batch.num_qo_heads * batch.head_dim * e
    lse = n_tok * batch.num_qo_heads * 4
    meta = 4 * (len(batch.kv_indices) + 2 * (batch.batch + 1) + batch.batch)
    return kv + qo + lse + meta


def prefill_flops(batch) -> float:
    """4 * D per visible (query, key) pair and qo head (QK^T and PV)."""
    tot = 0
    for q, k in zip(batch.qo_lens, batch.kv_lens):
        q, k = int(q), int(k)
        if batch.causal:
            vis = sum(max(0, min(k, i + k - q + 1)) for i in range(q))
        else:
            vis = q * k
        tot += vis
    return 4.0 * batch.head_dim * batch.num_qo_heads * tot


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def to_dev(batch, dev):
    return (batch.q.to(dev), batch.k_pages.to(dev), batch.v_pages.to(dev),
            torch.from_numpy(np.ascontiguousarray(batch.kv_indices, np.int32)).to(dev))


def time_kernel_only(pa, batch, dev_t, steps, warmup, qo=None):
    """Mean attention-kernel and merge-kernel time (ms) over `steps` runs of a fixed plan."""
    q, k, v, idx = dev_t
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    pa.plan(batch.kv_indptr, batch.last_page_len, qo_indptr=qo)
    for _ in range(warmup):
        pa.run_stages(q, k, v, idx, batch.sm_scale, out, lse)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        pa.run_stages(q, k, v, idx, batch.sm_scale, out, lse, events=ev[i])
    torch.cuda.synchronize()
    attn = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    merge = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    return attn, merge, out, lse


def run_ours(args, rank, world, local):
    import workloads
    from block_sparse_paged_gb300 import build
    build.build()
    import block_sparse_paged_gb300 as bsp

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    batch = workloads.batched_decode_bf16()
    nbytes = decode_bytes(batch)
    q, k, v, idx = to_dev(batch, dev)
    num_ctas = args.num_ctas or bsp.default_num_ctas(bsp.BSP_MODE_DECODE, local)
    # Two plan buffers (two workspaces) used in turn: step i's plan is copied on a
    # side stream while step i-1's kernel runs, and step i's kernel waits for
    # that copy; a buffer is rewritten only after the kernel that read it (two
    # steps back) has finished. Every step still plans on the host, copies its
    # plan and runs the kernel.
    pas = [bsp.PagedAttention("decode", batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size,
                              False, torch.bfloat16, max_batch=batch.batch, num_ctas=num_ctas, device=dev)
           for _ in range(2)]
    pa = pas[0]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup
    main, side = torch.cuda.current_stream(), torch.cuda.Stream(device=dev)
    run_done = [None, None]
    n_step = [0]

    def step(events=None):
        j = n_step[0] & 1
        n_step[0] += 1
        if run_done[j] is not None:
            side.wait_event(run_done[j])
        pas[j].plan(batch.kv_indptr, batch.last_page_len, stream=side)
        copied = torch.cuda.Event()
        copied.record(side)
        main.wait_event(copied)
        pas[j].run_stages(q, k, v, idx, batch.sm_scale, out, lse, stream=main, events=events)
        done = torch.cuda.Event()
        done.record(main)
        run_done[j] = done

    for _ in range(W):
        step()
    # Per-stage events go on one step in `every` (and always on the first): an event
    # between the attention kernel and the merge kernel keeps the merge from
    # being launched early (programmatic dependent launch), so the other steps
    # run without them; kernel durations are averaged over the sampled steps.
    every = 8
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for i in range(0, K, every)}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local).start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    barrier(world)
    torch.cuda.synchronize()
    t0.record()
    for i in range(K):
        step(ev.get(i))
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    step_ms = max_over_ranks(t0.elapsed_time(t1) / K, world)
    attn_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev.values())
    merge_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev.values())
    total_bytes = sum_over_ranks(float(nbytes), world)
    value = total_bytes / (step_ms * 1e-3) / 1e9

    pk, pk_src = peaks()
    achieved = nbytes / (attn_ms * 1e-3) / 1e9
    digest = kernel_digest(*DECODE_SOURCES)
    roofline = {"bound": "hbm", "kernel": "decode_bf16_kernel<128, TMA gather>", "achieved": round(achieved, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "peak_source": f"{pk_src} (STREAM-style copy)",
                "traffic": profile_traffic("decode_bf16_batched", digest),
                "algorithmic_bytes_per_launch": nbytes, "launch_ms": round(attn_ms, 5)}

    # host plan time alone (the planner's work plus queuing its one copy), after
    # the timed region: reported separately from the run time
    torch.cuda.synchronize()
    n_plan = min(200, K)
    tp = time.perf_counter()
    for _ in range(n_plan):
        pa.plan(batch.kv_indptr, batch.last_page_len)
    plan_ms_host = (time.perf_counter() - tp) * 1e3 / n_plan
    torch.cuda.synchronize()

    # end to end through the public API with host buffers
    e2e = run_e2e(bsp, batch, pa, K, W, dev, nbytes, world)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) values, numpy PCG64)",
        "config": {"workload": "batched paged decode, Llama-3-8B layer shape: 64 requests x 1 query, KV U{512..8192}, "
                               "page 16 (permuted pool), 32 qo / 8 kv heads, head_dim 128",
                   "name": WORKLOAD, "global_batch": batch.batch * world, "kv_tokens": int(batch.kv_lens.sum()),
                   "num_ctas": num_ctas, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 1.14 GB of KV per step vs 129 MB L2, no flush",
                   "step": "plan (host, one H2D copy) + decode kernel (split outputs merged inside it); two plan "
                           "buffers in turn, so step i's plan copy overlaps step i-1's kernel",
                   "algorithmic_bytes_per_step": nbytes, "merge_ms": round(merge_ms, 5),
                   "plan_ms_host": round(plan_ms_host, 5)},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": K,  # the decode kernel (split outputs are merged inside it)
        "clocks": clocks,
        "impl": "ours",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(batch, args.cpu_seconds)
    if rank == 0 and not args.no_secondary:
        del q, k, v, idx, out, lse
        torch.cuda.empty_cache()
        result["secondary"] = secondary(bsp, dev, args, pk)
    return result


def run_e2e(bsp, batch, pa, K, W, dev, nbytes, world):
    """Same metric through the public API, inputs copied host -> device from
    pinned memory and O, LSE copied back, every step."""
    hq = batch.q.pin_memory()
    hk = batch.k_pages.pin_memory()
    hv = batch.v_pages.pin_memory()
    hidx = torch.from_numpy(np.ascontiguousarray(batch.kv_indices, np.int32)).pin_memory()
    dq = torch.empty_like(hq, device=dev)
    dk = torch.empty_like(hk, device=dev)
    dv = torch.empty_like(hv, device=dev)
    didx = torch.empty_like(hidx, device=dev)
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty(hq.shape[:2], dtype=torch.float32).pin_memory()

    def step():
        pa.plan(batch.kv_indptr, batch.last_page_len)
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        didx.copy_(hidx, non_blocking=True)
        out, lse = pa.run(dq, dk, dv, didx, batch.sm_scale)
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    n = max(1, min(K, 10))
    for _ in range(max(1, min(W, 3))):
        step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(n):
        step()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1) / n, world)
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2 + hidx.numel() * 4 + pa.info.metadata_bytes
    d2h = ho.numel() * 2 + hl.numel() * 4
    total = sum_over_ranks(float(nbytes), world)
    return {"value": round(total / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "steps": n, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "KV pool, Q and page table copied from pinned host memory every step"}


def oracle_timed(batch, tok, head, seconds: float, threads: int = 0, k32=None, v32=None):
    """(repetitions, seconds) of the oracle, as it stands, over the selected
    (token, head) rows, repeated for about `seconds` (at least once). k32 / v32:
    the pools' values as float32 (default: the batch's own pools)."""
    import oracle
    if k32 is None:
        k32 = batch.k_pages.float().numpy()
    if v32 is None:
        v32 = batch.v_pages.float().numpy()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_rows_of(batch, tok, head, num_threads=threads, k_f32=k32, v_f32=v32)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            return reps, el


def all_rows(batch, n_req=None):
    """(token, head) of every output row of the first n_req requests (all by default)."""
    n_tok = int(batch.qo_indptr[batch.batch if n_req is None else n_req])
    return (np.repeat(np.arange(n_tok, dtype=np.int64), batch.num_qo_heads),
            np.tile(np.arange(batch.num_qo_heads, dtype=np.int32), n_tok))


def strided_rows(batch, stride: int, seed: int):
    """(token, head): every stride-th query position of each request and head,
    with a seeded phase per (request, head): a 1/stride sample of every request
    and head."""
    rng = np.random.default_rng(seed)
    toks, heads = [], []
    for b in range(batch.batch):
        q0, q1 = int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])
        for h in range(batch.num_qo_heads):
            sel = np.arange(q0 + int(rng.integers(stride)), q1, stride, dtype=np.int64)
            toks.append(sel)
            heads.append(np.full(sel.size, h, np.int32))
    return np.concatenate(toks), np.concatenate(heads)


def row_flops(batch, tok) -> float:
    """4 * D per visible (query, key) pair of the selected rows (one head each)."""
    b = np.searchsorted(batch.qo_indptr, tok, side="right") - 1
    qo, kv = batch.qo_lens[b], batch.kv_lens[b]
    if batch.causal:
        vis = np.clip(tok - batch.qo_indptr[b] + kv - qo + 1, 0, kv)
    else:
        vis = kv
    return 4.0 * batch.head_dim * float(np.sum(vis))


def cpu_baseline(batch, seconds: float):
    """The oracle, as it stands, on all host cores over the full workload,
    repeated for about `seconds`; then on one core over the first 4 requests."""
    import oracle
    tok, head = all_rows(batch)
    reps, el = oracle_timed(batch, tok, head, seconds)
    gbs = decode_bytes(batch) * reps / el / 1e9
    sub = workloads_sub(batch, 4)
    t1, h1 = all_rows(batch, 4)
    r1, e1 = oracle_timed(batch, t1, h1, seconds / 4, threads=1)
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": oracle.num_threads_available(), "kind": "oracle",
            "sample": f"full workload (64 requests x 32 heads), {reps} repetitions in {el:.1f} s, fp64",
            "one_core": {"value": round(decode_bytes(sub) * r1 / e1 / 1e9, 3), "unit": "GB/s", "cores": 1,
                         "sample": f"first 4 requests x 32 heads, {r1} repetitions in {e1:.1f} s, fp64"}}


def workloads_sub(batch, n_req):
    """The first n_req requests of a batch (same pools)."""
    import workloads
    return workloads.scaled(batch, qo_indptr=batch.qo_indptr[:n_req + 1], kv_indptr=batch.kv_indptr[:n_req + 1],
                            last_page_len=batch.last_page_len[:n_req])


def cpu_baseline_decode(batch, nbytes: float, seconds: float, what: str, k32=None, v32=None):
    """The oracle on all host cores over every output row of `batch`, repeated
    for about `seconds`; `nbytes` (the line's algorithmic bytes per run) per
    repetition gives the line's own unit."""
    import oracle
    tok, head = all_rows(batch)
    reps, el = oracle_timed(batch, tok, head, seconds, k32=k32, v32=v32)
    return {"value": round(nbytes * reps / el / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads_available(),
            "kind": "oracle", "sample": f"{what}: every output row, {reps} repetitions in {el:.1f} s, fp64"}


def cpu_baseline_prefill(batch, stride: int, seed: int, seconds: float):
    """The oracle on all host cores over a seeded 1/stride sample of the rows
    (every request and head), repeated for about `seconds`: GFLOP/s over the
    sampled rows' visible pairs."""
    import oracle
    tok, head = strided_rows(batch, stride, seed)
    reps, el = oracle_timed(batch, tok, head, seconds)
    fl = row_flops(batch, tok)
    return {"value": round(fl * reps / el / 1e9, 3), "unit": "GFLOP/s", "cores": oracle.num_threads_available(),
            "kind": "oracle",
            "sample": f"every {stride}th query position of every request and head (seeded phase, seed {seed}): "
                      f"{tok.size} rows, {fl:.3e} FLOP, {reps} repetitions in {el:.1f} s, fp64"}


def secondary(bsp, dev, args, pk):
    res = {}
    steps = max(5, min(args.steps, 50))
    warm = max(3, args.warmup)
    cpu = 0.0 if args.no_cpu_baseline else args.cpu_seconds / 2
    res["vector_sparse_decode"] = vector_sparse_decode(bsp, dev, steps, warm, pk, args.num_ctas, cpu)
    torch.cuda.empty_cache()
    res["ragged_causal_prefill"] = ragged_prefill(bsp, dev, steps, warm, pk, cpu)
    torch.cuda.empty_cache()
    res["vector_sparse_prefill"] = vector_sparse_prefill(bsp, dev, max(3, steps // 10), warm, pk, cpu)
    torch.cuda.empty_cache()
    res["bsr_prefill"] = bsr_prefill(bsp, dev, steps, warm, pk, cpu)
    torch.cuda.empty_cache()
    res["shared_prefix_decode"] = shared_prefix(bsp, dev, steps, warm, pk, cpu)
    res["fp8_kv_decode"] = fp8_decode(bsp, dev, steps, warm, pk, cpu)
    res["tiny_decode_f32"] = tiny_decode_f32(bsp, dev, steps, warm, pk)
    return res


def vector_sparse_decode(bsp, dev, steps, warm, pk, num_ctas=None, cpu_seconds=0.0):
    """Page size 1 (every token slot permuted) vs the same KV contiguous: GB/s
    of each and their ratio under the pages' LPT plan, and the permuted layout
    under the equal-share schedule for comparison (it evens out the 256 equal
    tiles on 152 CTAs, but adds split outputs and their fold)."""
    import workloads
    perm, cont = workloads.vector_sparse_decode_bf16()
    r = {}
    for tag, b, sched in (("permuted", perm, "lpt"), ("contiguous", cont, "lpt"), ("permuted_equal", perm, "equal")):
        C = num_ctas or bsp.default_num_ctas(bsp.BSP_MODE_DECODE, dev.index)
        pa = bsp.PagedAttention("decode", b.num_qo_heads, b.num_kv_heads, b.head_dim, 1, False, torch.bfloat16,
                                max_batch=b.batch, num_ctas=C, device=dev, schedule=sched)
        pa.plan(b.kv_indptr, b.last_page_len)
        q, k, v, idx = to_dev(b, dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        st = torch.cuda.Stream(device=dev)
        # one launch per run (split outputs are merged inside the kernel)
        ms = graph_time(lambda: pa.run(q, k, v, idx, b.sm_scale, out=out, lse=lse, stream=st), st, steps, warm)
        gbs = decode_bytes(b) / (ms * 1e-3) / 1e9
        r[tag] = {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "ms": round(ms, 4)}
        del pa, q, k, v, out, lse
        torch.cuda.empty_cache()
    r["permuted_over_contiguous"] = round(r["permuted"]["GB/s"] / r["contiguous"]["GB/s"], 4)
    if cpu_seconds > 0:
        r["cpu_baseline"] = cpu_baseline_decode(perm, decode_bytes(perm), cpu_seconds,
                                                "the permuted page-size-1 workload (32 requests x 64 heads)")
    r["workload"] = ("32 requests x 4096 tokens, page size 1 (131072 slots permuted), 64/8 heads, D 128, bf16; "
                     "the pages' LPT plan (permuted_equal: the equal-share plan); one launch per run, 10 per graph replay")
    r["roofline"] = {"bound": "hbm", "kernel": "decode_bf16_kernel<128, cp.async gather>",
                     "achieved": r["permuted"]["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": r["permuted"]["frac_of_hbm"], "peak_source": "measured (STREAM-style copy)",
                     "traffic": profile_traffic("decode_vector_sparse", kernel_digest(*DECODE_SOURCES)),
                     "algorithmic_bytes_per_launch": decode_bytes(perm)}
    return r


def bsr_prefill(bsp, dev, steps, warm, pk, cpu_seconds=0.0):
    """General BSR prefill (row blocks of 64 queries, 16-token column blocks,
    25% density), graph-timed."""
    import workloads
    b = workloads.bsr_prefill_bf16()
    pa = bsp.PagedAttention("prefill", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, False,
                            torch.bfloat16, max_batch=b.batch, max_qo_tokens=int(b.qo_indptr[-1]), device=dev)
    pa.plan(b.kv_indptr, b.last_page_len, qo_indptr=b.qo_indptr)
    q, k, v, idx = to_dev(b, dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)
    # a run is the attention kernel and the merge of split outputs (none here)
    ms = graph_time(lambda: pa.run(q, k, v, idx, b.sm_scale, out=out, lse=lse, stream=st), st, steps, warm)
    fl = prefill_flops(b)
    tf = fl / (ms * 1e-3) / 1e12
    r = {"TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
         "ms": round(ms, 4), "flops": fl,
         "workload": "general BSR: 32 row blocks of 64 queries, 512 column blocks of 16 tokens, "
                     "25% block density, 32/8 heads, D 128, bf16, non-causal; 10 runs per graph replay",
         "roofline": {"bound": "tensor", "kernel": "prefill_kernel<TMA>", "achieved": round(tf, 1),
                      "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(tf / pk["bf16_tflops"], 4),
                      "peak_source": "measured (cuBLAS bf16 burst)",
                      "traffic": profile_traffic("prefill_bsr", kernel_digest(*PREFILL_SOURCES)),
                      "algorithmic_flops_per_launch": fl}}
    del pa, q, k, v, out, lse
    if cpu_seconds > 0:
        r["cpu_baseline"] = cpu_baseline_prefill(b, 8, 7, cpu_seconds)
    return r


def tiny_decode_f32(bsp, dev, steps, warm, pk):
    """The tiny fp32 paged decode (3 requests, KV 10 / 3 / 7, page 4, 4/2 heads,
    D 64): latency of one run (graph-timed), correctness-sized."""
    import workloads
    b = workloads.tiny_decode_f32()
    pa = bsp.PagedAttention("decode", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, False,
                            torch.float32, max_batch=b.batch, device=dev)
    pa.plan(b.kv_indptr, b.last_page_len)
    q, k, v, idx = to_dev(b, dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)
    ms = graph_time(lambda: pa.run(q, k, v, idx, b.sm_scale, out=out, lse=lse, stream=st), st, steps, warm)
    return {"us": round(ms * 1e3, 2), "bytes": decode_bytes(b), "kernel": "decode_f32_kernel",
            "workload": "3 requests, KV 10 / 3 / 7, page 4 (16-page permuted pool), 4/2 heads, D 64, fp32; "
                        "10 runs per graph replay"}


def ragged_prefill(bsp, dev, steps, warm, pk, cpu_seconds=0.0):
    """The ragged causal prefill workload, kernel-only timing with a roofline.
    Planned for two LPT queues per CTA (each CTA runs two consecutive queues):
    swept on GB300 (graph-timed, alpha 2), 152 / 304 / 456 queues 279.4 /
    273.8 / 283.0 us; no tile is split at any of them."""
    import workloads
    b = workloads.ragged_causal_prefill_bf16()
    C = 2 * torch.cuda.get_device_properties(dev).multi_processor_count
    pa = bsp.PagedAttention("prefill", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, True,
                            torch.bfloat16, max_batch=b.batch, max_qo_tokens=int(b.qo_indptr[-1]), num_ctas=C,
                            device=dev)
    dev_t = to_dev(b, dev)
    attn, merge, out, lse = time_kernel_only(pa, b, dev_t, steps, warm, qo=b.qo_indptr)
    fl = prefill_flops(b)
    tf = fl / ((attn + merge) * 1e-3) / 1e12
    ka = fl / (attn * 1e-3) / 1e12
    clk = clocks_while(lambda: pa.run_stages(*dev_t, b.sm_scale, out, lse), 1.5, dev.index or 0)
    del pa
    cpu = cpu_baseline_prefill(b, 8, 4, cpu_seconds) if cpu_seconds > 0 else None
    return {"cpu_baseline": cpu,
        "TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4), "flops": fl,
        "attn_ms": round(attn, 4), "merge_ms": round(merge, 4),
        "workload": "16 requests, qo = kv ~ U{128..2048}, page 16 permuted, 32/8 heads, D 128, bf16, causal; "
                    "plan of 2 queues per CTA", "plan_queues": C,
        "clocks_sustained": clk,
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": round(ka, 1),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(ka / pk["bf16_tflops"], 4),
                     "peak_source": "measured (cuBLAS bf16 burst; the kernel is timed alone)",
                     "traffic": profile_traffic("prefill_ragged_causal", kernel_digest(*PREFILL_SOURCES)),
                     "algorithmic_flops_per_launch": fl}}


def graph_time(run, st, steps, warm, reps=10):
    """Mean time (ms) of one run() call, launched `reps` times per CUDA graph
    replay so that the host's per-call cost stays out of the kernel time."""
    with torch.cuda.stream(st):
        for _ in range(warm):
            run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for _ in range(reps):
            run()
    graph.replay()
    n_rep = max(1, steps // reps)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    torch.cuda.synchronize()
    ev[0].record()  # replay() launches on the current stream
    for i in range(n_rep):
        graph.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    ms = statistics.mean(ev[i].elapsed_time(ev[i + 1]) for i in range(n_rep)) / reps
    del graph
    return ms


def fp8_decode(bsp, dev, steps, warm, pk, cpu_seconds=0.0):
    """The batched decode workload with e4m3 K / V pools (one scale each):
    algorithmic bytes as for bf16 but one byte per K / V element."""
    import workloads
    b = workloads.batched_decode_bf16()
    f8 = workloads.fp8_kv(b)
    pa = bsp.PagedAttention("decode", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, False,
                            torch.bfloat16, max_batch=b.batch, device=dev)
    pa.plan(b.kv_indptr, b.last_page_len)
    q = b.q.to(dev)
    k = f8.k8.to(dev).view(torch.float8_e4m3fn)
    v = f8.v8.to(dev).view(torch.float8_e4m3fn)
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_indices, np.int32)).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    st = torch.cuda.Stream(device=dev)

    def run():
        pa.run(q, k, v, idx, b.sm_scale, out=out, lse=lse, k_scale=f8.k_scale, v_scale=f8.v_scale, stream=st)
    ms = graph_time(run, st, steps, warm)
    kv_tokens = int(b.kv_lens.sum())
    nbytes = decode_bytes(b) - kv_tokens * b.num_kv_heads * b.head_dim * 2 * (esize(b) - 1)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del pa, q, k, v
    torch.cuda.empty_cache()
    cpu = {}
    if cpu_seconds > 0:
        import oracle.fp8
        # the oracle over the values the codes stand for (k_scale * value(code))
        k32 = oracle.fp8.dequantize(f8.k8.numpy(), f8.k_scale).astype(np.float32)
        v32 = oracle.fp8.dequantize(f8.v8.numpy(), f8.v_scale).astype(np.float32)
        cpu["cpu_baseline"] = cpu_baseline_decode(b, nbytes, cpu_seconds, "the e4m3 batched decode (64 requests x "
                                                  "32 heads, codes decoded once outside the timing)", k32=k32, v32=v32)
    return {**cpu, "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "ms": round(ms, 4),
            "bytes": nbytes, "tokens_per_s": round(b.batch / (ms * 1e-3), 1),
            "workload": "batched decode (64 requests, KV ~ U{512..8192}, page 16 permuted, 32/8 heads, D 128), "
                        "K / V e4m3 with one scale per pool, q / o bf16; one launch per step, 10 per graph replay",
            "roofline": {"bound": "hbm", "kernel": "decode_bf16_kernel<128, TMA gather, e4m3>",
                         "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm_gbs"], 4), "peak_source": "measured (STREAM-style copy)",
                         "traffic": profile_traffic("decode_fp8_batched", kernel_digest(*DECODE_SOURCES)),
                         "algorithmic_bytes_per_launch": nbytes}}


def vector_sparse_prefill(bsp, dev, steps, warm, pk, cpu_seconds=0.0):
    """One 32768-token causal prefill with page size 1, once on permuted slots and
    once contiguous, each planned with a gather region for its page table (the
    pages are copied into the workspace in table order, then read by TMA; the
    copy is inside the timed run), and once permuted without a region (16-byte
    cp.async gather): TFLOP/s of each, their ratios, and the same KV as
    128-token pages (TMA page gather, no copy)."""
    import workloads
    import dataclasses
    perm, cont = workloads.vector_sparse_prefill_bf16()
    n = int(cont.kv_indptr[-1])
    # the same contiguous KV seen as 128-token pages: the dense-layout reference (TMA gather)
    dense = dataclasses.replace(cont, name="vector_sparse_prefill_bf16_pages128", page_size=128,
                                kv_indptr=np.array([0, n // 128], np.int32), kv_indices=np.arange(n // 128, dtype=np.int32),
                                last_page_len=np.array([128], np.int32),
                                k_pages=cont.k_pages.reshape(n // 128, 128, cont.num_kv_heads, cont.head_dim),
                                v_pages=cont.v_pages.reshape(n // 128, 128, cont.num_kv_heads, cont.head_dim))
    fl = prefill_flops(perm)
    r = {}
    for tag, b, region in (("permuted", perm, n), ("contiguous", cont, n), ("permuted_cp_async", perm, 0),
                           ("contiguous_pages128", dense, 0)):
        pa = bsp.PagedAttention("prefill", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, True,
                                torch.bfloat16, max_batch=1, max_qo_tokens=int(b.qo_indptr[-1]), device=dev,
                                max_gather_pages=region)
        attn, merge, _, _ = time_kernel_only(pa, b, to_dev(b, dev), steps, warm, qo=b.qo_indptr)
        tf = fl / ((attn + merge) * 1e-3) / 1e12
        r[tag] = {"TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                  "attn_ms": round(attn, 4), "merge_ms": round(merge, 4)}
        del pa
        torch.cuda.empty_cache()
    r["permuted_over_contiguous"] = round(r["permuted"]["TFLOP/s"] / r["contiguous"]["TFLOP/s"], 4)
    r["page1_over_pages128"] = round(r["permuted"]["TFLOP/s"] / r["contiguous_pages128"]["TFLOP/s"], 4)
    r["flops"] = fl
    r["workload"] = ("1 request, qo = kv = 32768, causal, page size 1 (slots permuted / contiguous; page copy into "
                     "the workspace + TMA, or cp.async gather) and the same KV as 128-token pages (TMA page gather), "
                     "32/8 heads, D 128, bf16")
    r["pages_context"] = "FA3 template on H100: 532 (page 1) vs 627 (contiguous) TFLOP/s"
    if cpu_seconds > 0:
        r["cpu_baseline"] = cpu_baseline_prefill(perm, 128, 6, cpu_seconds)
    return r


def shared_prefix_bytes(sp) -> int:
    """Prefix KV once, every suffix's KV, Q, O, LSE and both page tables."""
    e = 2
    kvrow = sp.full.num_kv_heads * sp.full.head_dim * e * 2
    n_tok = int(sp.full.qo_indptr[-1])
    qo = 2 * n_tok * sp.full.num_qo_heads * sp.full.head_dim * e
    lse = n_tok * sp.full.num_qo_heads * 4
    meta = 4 * (len(sp.prefix.kv_indices) + len(sp.suffix.kv_indices) + 3 * (sp.full.batch + 1))
    return sp.prefix_len * kvrow + int(sp.suffix_lens.sum()) * kvrow + qo + lse + meta


def shared_prefix_split(bsp, dev, prefix_tiles: int = 8):
    """CTAs for the prefix view (prefill kernel); the rest run the suffix view
    concurrently. A multiple of the prefix view's output tiles (8: one 256-row
    tile per kv head) gives every CTA one equal chunk of the shared pages;
    among those, the one nearest a fifth of the SMs. Swept on this workload
    (GB300, 152 SMs): 16 / 24 / 32 / 40 / 48 CTAs 89.5 / 73.3 / 68.3 / 73.3 /
    74.8 us per step; counts that split the chunks unevenly are slower (20:
    86.4, 51: 77.6)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    c = max(prefix_tiles, round(sms / 5 / prefix_tiles) * prefix_tiles)
    return min(c, sms - 8), sms


def shared_prefix(bsp, dev, steps, warm, pk, cpu_seconds=0.0):
    """Composable decode: prefix view on the prefill kernel (all 64 queries as one
    row block over the shared pages) and suffix view on the decode kernel, run
    concurrently on two streams over disjoint SM counts (their plans are made
    for those CTA counts), then merge_state. The step is captured in a CUDA
    graph (host launch costs stay out) and replayed."""
    import workloads
    sp = workloads.shared_prefix_decode_bf16()
    q = sp.full.q.to(dev)
    k = sp.full.k_pages.to(dev)
    v = sp.full.v_pages.to(dev)
    ip = torch.from_numpy(sp.prefix.kv_indices).to(dev)
    isf = torch.from_numpy(sp.suffix.kv_indices).to(dev)
    c_pre, sms = shared_prefix_split(bsp, dev)
    pre = bsp.PagedAttention("prefill", 32, 8, 128, sp.full.page_size, False, torch.bfloat16, max_batch=1,
                             max_qo_tokens=int(sp.prefix.qo_indptr[-1]), num_ctas=c_pre, device=dev)
    suf = bsp.PagedAttention("decode", 32, 8, 128, sp.full.page_size, False, torch.bfloat16,
                             max_batch=sp.suffix.batch, num_ctas=sms - c_pre, device=dev)
    pre.plan(sp.prefix.kv_indptr, sp.prefix.last_page_len, qo_indptr=sp.prefix.qo_indptr)
    suf.plan(sp.suffix.kv_indptr, sp.suffix.last_page_len)
    torch.cuda.synchronize()
    o1 = torch.empty_like(q)
    o2 = torch.empty_like(q)
    l1 = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    l2 = torch.empty_like(l1)
    out = torch.empty_like(q)
    lse = torch.empty_like(l1)
    main, s_pre, s_suf = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def step():
        s_pre.wait_stream(main)
        s_suf.wait_stream(main)
        pre.run(q, k, v, ip, sp.full.sm_scale, out=o1, lse=l1, stream=s_pre)
        suf.run(q, k, v, isf, sp.full.sm_scale, out=o2, lse=l2, stream=s_suf)
        main.wait_stream(s_pre)
        main.wait_stream(s_suf)
        bsp.merge_state(o1, l1, o2, l2, out=out, lse_out=lse, stream=main)

    with torch.cuda.stream(main):
        for _ in range(warm):
            step()
    torch.cuda.synchronize()
    reps = 10
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=main):
        for _ in range(reps):
            step()
    graph.replay()
    n_rep = max(1, steps // reps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n_rep):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (n_rep * reps)
    nbytes = shared_prefix_bytes(sp)
    gbs = nbytes / (ms * 1e-3) / 1e9
    n, P, S = sp.full.batch, sp.prefix_len, float(sp.suffix_lens.mean())
    ratio = n * (P + S) / (P + n * S)
    del graph
    cpu = {}
    if cpu_seconds > 0:
        # the oracle computes each request over its whole KV (prefix and suffix),
        # timed against the same prefix-once bytes as the line
        cpu["cpu_baseline"] = cpu_baseline_decode(sp.full, nbytes, cpu_seconds,
                                                  "each of the 64 requests over its prefix and suffix")
    return {**cpu, "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "ms": round(ms, 4),
            "algorithmic_bytes": nbytes, "launches_per_step": 4, "ctas_prefix_view": c_pre,
            "ctas_suffix_view": sms - c_pre, "eq15_traffic_ratio": round(ratio, 3),
            "workload": "64 decode requests sharing an 8192-token prefix, suffixes U{64..1024} and one 32768 "
                        "outlier, page 16, 32/8 heads, D 128, bf16; prefix and suffix views concurrent on two "
                        "streams, 10 steps per CUDA graph replay"}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    import oracle
    import workloads
    if rank != 0:
        return None
    oracle.build()
    batch = workloads.batched_decode_bf16()
    k32 = batch.k_pages.float().numpy()
    v32 = batch.v_pages.float().numpy()
    # each step: the first 16 requests, all 32 heads (a bounded sample of the workload)
    nreq = 16
    tok = np.repeat(np.arange(nreq, dtype=np.int64), batch.num_qo_heads)
    head = np.tile(np.arange(batch.num_qo_heads, dtype=np.int32), nreq)
    sub = workloads.scaled(batch, qo_indptr=batch.qo_indptr[:nreq + 1], kv_indptr=batch.kv_indptr[:nreq + 1],
                           last_page_len=batch.last_page_len[:nreq])
    nbytes = decode_bytes(sub)
    for _ in range(args.warmup):
        oracle.attention_rows_of(batch, tok, head, k_f32=k32, v_f32=v32)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_rows_of(batch, tok, head, k_f32=k32, v_f32=v32)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = nbytes / (ms * 1e-3) / 1e9
    cores = oracle.num_threads_available()
    return {"metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) values, numpy PCG64)",
            "config": {"workload": "batched paged decode, Llama-3-8B layer shape (first 16 of the 64 requests per step)",
                       "name": WORKLOAD, "sample_requests": nreq},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {nreq} requests x 32 heads per step, fp64 C oracle"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# secondary workloads that `--case` runs alone (profiling)
CASES = {"ragged_causal_prefill": ragged_prefill, "fp8_kv_decode": fp8_decode, "shared_prefix_decode": shared_prefix,
         "vector_sparse_prefill": vector_sparse_prefill, "vector_sparse_decode": vector_sparse_decode,
         "bsr_prefill": bsr_prefill, "tiny_decode_f32": tiny_decode_f32}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--num-ctas", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="run one secondary workload alone (steps / warmup as given) and print its line; "
                         "for profiling")
    args = ap.parse_args(argv)
    if args.case:
        from block_sparse_paged_gb300 import build
        build.build()
        import block_sparse_paged_gb300 as bsp
        dev = torch.device("cuda", 0)
        print(json.dumps({args.case: CASES[args.case](bsp, dev, args.steps, args.warmup, peaks()[0])}), flush=True)
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
