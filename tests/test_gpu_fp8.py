"""Decode over an e4m3 KV cache (FlashInfer: A Customizable Attention Engine
for LLM Serving, App. G.4 Table 8, the e4m3 rows) against the oracle run on
the values the codes stand for (oracle.fp8: k_scale * value(code))."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare, lib, timed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    return lib()


def run_fp8(bsp, b, f8, num_ctas=None, repeats=1, sink=None):
    pa = bsp.PagedAttention("decode", b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, False,
                            torch.bfloat16, max_batch=b.batch, num_ctas=num_ctas, window_left=b.window_left,
                            logits_soft_cap=b.soft_cap)
    pa.plan(b.kv_indptr, b.last_page_len)
    q = b.q.cuda()
    k = f8.k8.cuda().view(torch.float8_e4m3fn)
    v = f8.v8.cuda().view(torch.float8_e4m3fn)
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_indices, np.int32)).cuda()
    sk = None if sink is None else torch.tensor(sink, dtype=torch.float32, device="cuda")
    for _ in range(repeats):
        out, lse = pa.run(q, k, v, idx, b.sm_scale, k_scale=f8.k_scale, v_scale=f8.v_scale, sink=sk)
    torch.cuda.synchronize()
    return out, lse, pa


def oracle_kv(f8):
    return (oracle.fp8.dequantize(f8.k8.numpy(), f8.k_scale), oracle.fp8.dequantize(f8.v8.numpy(), f8.v_scale))


CASES = [
    # (seed, kv lens, H_qo, H_kv, page, num_ctas, window, cap)
    (101, [3000, 17, 900, 4100, 1, 250, 64, 65], 32, 8, 16, 29, -1, 0.0),   # splits, ragged tails
    (102, [5000, 33, 129], 32, 8, 8, 17, -1, 0.0),                         # page 8 (box of 8 rows)
    (103, [2048, 1000, 7], 16, 4, 32, 11, -1, 0.0),
    (104, [4000, 300], 64, 8, 64, 9, -1, 0.0),                             # g = 8, page 64
    (105, [6000, 130, 2], 32, 2, 128, 23, -1, 0.0),                        # g = 16, page 128 (two boxes)
    (106, [3000, 900, 4100], 32, 8, 16, 13, 700, 1.5),                     # window and soft-cap
    (107, [0, 40, 0, 1], 32, 8, 16, 5, -1, 0.0),                           # empty requests
]


@pytest.mark.parametrize("case", CASES, ids=[f"fp8_{c[0]}" for c in CASES])
def test_fp8_decode(bsp, case):
    seed, kv, hq, hk, ps, C, w, cap = case
    b = workloads.paged_batch(seed, [1] * len(kv), kv, hq, hk, 128, ps, "bf16", extra_pages=3)
    b.window_left, b.soft_cap = w, cap
    f8 = workloads.fp8_kv(b)
    kd, vd = oracle_kv(f8)
    O, L = oracle.attention_of(b, k=kd, v=vd)
    out, lse, pa = run_fp8(bsp, b, f8, num_ctas=C)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_fp8_sink(bsp):
    """Attention sink on the e4m3 path: split outputs (fused merge) and an empty request."""
    b = workloads.paged_batch(112, [1] * 4, [3000, 0, 700, 4100], 32, 8, 128, 16, "bf16", extra_pages=1)
    f8 = workloads.fp8_kv(b)
    sk = np.random.default_rng(112).uniform(-2.0, 4.0, size=32)
    kd, vd = oracle_kv(f8)
    O, L = oracle.attention_of(b, k=kd, v=vd, sink=sk)
    out, lse, _ = run_fp8(bsp, b, f8, num_ctas=19, sink=sk)
    compare(out, lse, O, L, "bf16")


def test_fp8_scales_are_applied(bsp):
    """Scaling K by 2 doubles every score and V by 3 triples every output: the
    same codes with other scales against the oracle with those scales."""
    b = workloads.paged_batch(108, [1] * 3, [700, 64, 2000], 32, 8, 128, 16, "bf16", extra_pages=1)
    f8 = workloads.fp8_kv(b)
    f8.k_scale *= 2.0
    f8.v_scale *= 3.0
    kd, vd = oracle_kv(f8)
    O, L = oracle.attention_of(b, k=kd, v=vd)
    out, lse, _ = run_fp8(bsp, b, f8, num_ctas=7)
    compare(out, lse, O, L, "bf16")


def test_fp8_full_size_decode(bsp):
    """The Llama-3-8B-shaped batched decode (batch 64, KV up to 8192, page 16)
    with e4m3 K / V: every output row against the oracle; run twice on one plan
    (the in-kernel merge resets its counters)."""
    b = workloads.batched_decode_bf16()
    f8 = workloads.fp8_kv(b)
    out, lse, pa = run_fp8(bsp, b, f8, repeats=2)
    kd, vd = oracle_kv(f8)
    (O, L), t = timed(oracle.attention_of, b, k=kd, v=vd)
    compare(out, lse, O, L, "bf16", oracle_s=t)
    assert pa.check_device_error() == 0


def test_fp8_rejects_bad_scales_and_shapes(bsp):
    b = workloads.paged_batch(109, [1, 1], [100, 50], 32, 8, 128, 16, "bf16")
    f8 = workloads.fp8_kv(b)
    f8.k_scale = 0.0
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        run_fp8(bsp, b, f8)
    b64 = workloads.paged_batch(110, [1, 1], [100, 50], 32, 8, 64, 16, "bf16")
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        run_fp8(bsp, b64, workloads.fp8_kv(b64))
    b4 = workloads.paged_batch(111, [1, 1], [100, 50], 32, 8, 128, 4, "bf16")
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        run_fp8(bsp, b4, workloads.fp8_kv(b4))


def test_fp8_graph_replay_with_sink(bsp):
    """An e4m3 decode run with sinks captured in a CUDA graph, then replayed
    after a re-plan of other requests loaded into the same pools (one scale
    pair for both, as the captured launch holds the scales): both replays
    match the oracle."""
    a = workloads.paged_batch(113, [1] * 5, [3000, 17, 900, 0, 2200], 32, 8, 128, 16, "bf16", extra_pages=3)
    bb = workloads.paged_batch(114, [1] * 5, [50, 4000, 1, 700, 1300], 32, 8, 128, 16, "bf16", extra_pages=3)

    def amax(t):
        return float(torch.nan_to_num(t.float(), nan=0.0).abs().max())
    ks = max(amax(a.k_pages), amax(bb.k_pages)) / 448.0
    vs = max(amax(a.v_pages), amax(bb.v_pages)) / 448.0
    codes = {id(b): ((b.k_pages.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8),
                     (b.v_pages.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)) for b in (a, bb)}
    sk = np.random.default_rng(113).uniform(-2.0, 4.0, size=32)
    pool = max(a.k_pages.shape[0], bb.k_pages.shape[0])
    k8 = torch.zeros((pool, 16, 8, 128), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    q = torch.empty_like(a.q, device="cuda")
    idx = torch.zeros(1024, dtype=torch.int32, device="cuda")
    sink = torch.tensor(sk, dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")

    def load(b):
        kc, vc = codes[id(b)]
        k8[: kc.shape[0]].copy_(kc)
        v8[: vc.shape[0]].copy_(vc)
        q.copy_(b.q)
        idx[: len(b.kv_indices)].copy_(torch.from_numpy(np.ascontiguousarray(b.kv_indices, np.int32)))

    pa = bsp.PagedAttention("decode", 32, 8, 128, 16, False, torch.bfloat16, max_batch=5, num_ctas=19)
    kf, vf = k8.view(torch.float8_e4m3fn), v8.view(torch.float8_e4m3fn)

    def run():
        pa.run(q, kf, vf, idx, a.sm_scale, out=out, lse=lse, k_scale=ks, v_scale=vs, sink=sink)
    load(a)
    pa.plan(a.kv_indptr, a.last_page_len)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()  # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for b in (a, bb):
        if b is bb:
            load(bb)
            pa.plan(bb.kv_indptr, bb.last_page_len)
        g.replay()
        torch.cuda.synchronize()
        kc, vc = codes[id(b)]
        O, L = oracle.attention_of(b, k=oracle.fp8.dequantize(kc.numpy(), ks),
                                   v=oracle.fp8.dequantize(vc.numpy(), vs), sink=sk)
        compare(out, lse, O, L, "bf16")
