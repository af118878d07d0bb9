"""Decode path on the GPU through the C ABI, element by element against the
oracle on the same seeded inputs."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from block_sparse_paged_gb300 import _native as N
from gpu_helpers import (compare, lib, oracle_full, run_batch, timed, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    return lib()


def test_tiny_decode_f32(bsp):
    """3 requests, KV 10/3/7, page 4, 16-page permuted pool with NaN in unused
    pages and page tails, 4/2 heads, head_dim 64, fp32, sm_scale 1/8."""
    b = workloads.tiny_decode_f32()
    O, L = oracle_full(b)
    for C in (1, 3, 64):
        out, lse, _ = run_batch(bsp, b, num_ctas=C)
        compare(out, lse, O, L, "f32")


CASES = [
    # (seed, kv lens, H_qo, H_kv, D, page, num_ctas)
    (1, [1, 64, 65, 127, 200, 0, 3000], 32, 8, 128, 16, 7),
    (2, [5, 17, 64, 1000, 4097], 8, 8, 128, 1, 5),
    (3, [33, 300, 2, 511, 1500, 64], 16, 2, 128, 3, 11),
    (4, [700, 1, 129, 4000], 16, 1, 128, 16, 3),
    (5, [100, 257, 0, 63], 4, 2, 64, 4, 6),
    (6, [2048, 1024, 17], 32, 4, 64, 1, 400),
    (7, [12345, 5, 999], 32, 8, 128, 32, 2),
    (8, [513, 31, 64, 2000], 32, 2, 64, 8, 13),        # g = 16, D = 64, 8-row page boxes
    (9, [129, 4000, 1], 32, 8, 128, 64, 9),            # 64-token pages: one box per stage half
    (10, [300, 5000, 260, 17], 64, 8, 128, 256, 21),   # 256-token pages: four boxes per page
    (11, [4096, 130, 3, 1, 700], 64, 8, 128, 1, 19),   # page 1, g = 8, ragged stage tails
    (12, [1000, 37, 2500, 6], 32, 8, 128, 12, 9),      # 12-token pages (not a power of two): cp.async
    (13, [513, 2, 3001], 8, 2, 64, 2, 7),              # D = 64, 2-token pages
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_random_bf16_decode(bsp, case):
    seed, kv, hq, hk, D, ps, C = case
    b = workloads.paged_batch(seed, np.ones(len(kv), int), kv, hq, hk, D, ps, "bf16", extra_pages=3)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=C)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_batched_decode_full_size(bsp):
    """Llama-3-8B-shaped batch at full size (64 requests, KV U{512..8192}, page
    16), every output row against the oracle, with the bench's CTA count."""
    b = workloads.batched_decode_bf16()
    out, lse, pa = run_batch(bsp, b)
    (O, L), t = timed(oracle_full, b)
    compare(out, lse, O, L, "bf16", oracle_s=t)
    # run twice: bitwise identical (fixed plan, fixed reduction order)
    q, k, v, idx = to_dev(b)
    out2, lse2 = pa.run(q, k, v, idx, b.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_vector_sparse_permuted_equals_contiguous(bsp):
    """Page size 1, every slot permuted, 64/8 heads: the permuted and the
    contiguous layouts give bitwise-equal outputs; every output row matches the
    oracle."""
    perm, cont = workloads.vector_sparse_decode_bf16()
    out_p, lse_p, _ = run_batch(bsp, perm)
    out_c, lse_c, _ = run_batch(bsp, cont)
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    (O, L), t = timed(oracle_full, perm)
    compare(out_p, lse_p, O, L, "bf16", oracle_s=t)


def test_vector_sparse_equal_shares(bsp):
    """The page-size-1 decode with the equal-share schedule (every CTA 6898-6899
    tokens in at most 3 items, most tiles split): permuted and contiguous layouts
    bitwise equal, every output row against the oracle."""
    perm, cont = workloads.vector_sparse_decode_bf16()
    out_p, lse_p, pa = run_batch(bsp, perm, schedule="equal")
    assert pa.info.num_merges > 0
    out_c, lse_c, _ = run_batch(bsp, cont, schedule="equal")
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    (O, L), t = timed(oracle_full, perm)
    compare(out_p, lse_p, O, L, "bf16", oracle_s=t)
    assert pa.check_device_error() == 0


@pytest.mark.parametrize("case", CASES[:8], ids=[f"equal{c[0]}" for c in CASES[:8]])
def test_random_equal_share_decode(bsp, case):
    """Random decode batches under the equal-share schedule (splits inside
    requests at page boundaries, empty requests, several items per CTA)."""
    seed, kv, hq, hk, D, ps, C = case
    b = workloads.paged_batch(seed, np.ones(len(kv), int), kv, hq, hk, D, ps, "bf16", extra_pages=3)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=C, schedule="equal")
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


@pytest.mark.parametrize("ps,D", [(16, 128), (8, 64), (64, 128)])
def test_tma_gather_equals_cp_async_gather(bsp, ps, D):
    """Pages of 8 or more tokens are gathered by TMA page boxes when the pool
    size is known, by 16-byte cp.async copies when it is not (num_pages 0):
    the two loaders fill the same swizzled tiles, so the outputs are bitwise
    equal; both match the oracle."""
    import ctypes
    b = workloads.paged_batch(50 + ps, np.ones(5, int), [3001, 17, 1, 640, 129], 32, 8, D, ps, "bf16",
                              extra_pages=3)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=23)
    compare(out, lse, O, L, "bf16")
    q, k, v, idx = to_dev(b)
    out0 = torch.empty_like(q)
    lse0 = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    rc = pa.lib.bsp_decode_run(ctypes.byref(pa.info), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                               ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(idx.data_ptr()), 0,
                               ctypes.c_float(b.sm_scale), ctypes.c_void_p(out0.data_ptr()),
                               ctypes.c_void_p(lse0.data_ptr()), ctypes.c_void_p(pa.workspace.data_ptr()),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert pa.check_device_error() == 0
    assert torch.equal(out.cuda(), out0) and torch.equal(lse.cuda(), lse0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_many_slot_folds(bsp, dtype):
    """Plans with many chunks per CTA: outputs split into more than 8 partial
    states, so the in-kernel fold takes its batches of 8 with rescaling to the
    running maximum (bf16 and fp32 kernels); against the oracle."""
    b = workloads.paged_batch(61, np.ones(5, int), [6000, 2500, 17, 900, 4100], 32, 8, 128, 16, dtype,
                              extra_pages=3)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=11, chunks_per_cta=16)
    q_, items, merges = pa.plan_arrays()
    assert int(merges["n_slots"].max()) > 8
    compare(out, lse, O, L, dtype)
    assert pa.check_device_error() == 0


def test_shared_prefix_full_view_decode(bsp):
    """The shared-prefix batch read without composition (every request over
    prefix + suffix pages), including the 32768-token outlier; every output row."""
    sp = workloads.shared_prefix_decode_bf16()
    out, lse, _ = run_batch(bsp, sp.full)
    (O, L), t = timed(oracle_full, sp.full)
    compare(out, lse, O, L, "bf16", oracle_s=t)


def test_cuda_graph_replay_with_new_plan(bsp):
    """Capture one run, then re-plan with other lengths into the same workspace
    and replay: the replay equals an eager run of the new plan."""
    hq, hk, D, ps = 32, 8, 128, 16
    a = workloads.paged_batch(21, np.ones(6, int), [100, 2000, 5, 700, 64, 3000], hq, hk, D, ps, "bf16", extra_pages=40)
    bb = workloads.paged_batch(22, np.ones(6, int), [3000, 1, 64, 65, 2500, 10], hq, hk, D, ps, "bf16", extra_pages=40)
    pa = bsp.PagedAttention("decode", hq, hk, D, ps, False, torch.bfloat16, max_batch=6, num_ctas=24)
    pool = max(a.k_pages.shape[0], bb.k_pages.shape[0])
    q = torch.empty_like(a.q, device="cuda")
    k = torch.empty((pool,) + tuple(a.k_pages.shape[1:]), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    idx = torch.zeros(8192, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")

    def load(batch):
        q.copy_(batch.q)
        k[: batch.k_pages.shape[0]].copy_(batch.k_pages)
        v[: batch.v_pages.shape[0]].copy_(batch.v_pages)
        idx[: len(batch.kv_indices)].copy_(torch.from_numpy(batch.kv_indices))

    load(a)
    pa.plan(a.kv_indptr, a.last_page_len)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.run(q, k, v, idx, a.sm_scale, out=out, lse=lse)  # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.run(q, k, v, idx, a.sm_scale, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    O, L = oracle_full(a)
    compare(out, lse, O, L, "bf16")
    load(bb)
    pa.plan(bb.kv_indptr, bb.last_page_len)
    g.replay()
    torch.cuda.synchronize()
    O, L = oracle_full(bb)
    compare(out, lse, O, L, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_state_of_split_attention(bsp, dtype):
    """Two attention states over disjoint page ranges of the same requests,
    merged on the GPU, equal attention over all pages (oracle)."""
    b = workloads.paged_batch(30, np.ones(8, int), [40, 33, 100, 17, 64, 250, 9, 128], 16, 4, 128, 4, dtype,
                              extra_pages=5)
    half = [(int(b.kv_indptr[i]) + int(b.kv_indptr[i + 1])) // 2 for i in range(b.batch)]
    first = workloads.scaled(b, kv_indptr=np.array([0] + [h - int(b.kv_indptr[i]) for i, h in enumerate(half)]).cumsum().astype(np.int32),
                             kv_indices=np.concatenate([b.kv_indices[b.kv_indptr[i]:half[i]] for i in range(b.batch)]).astype(np.int32),
                             last_page_len=np.full(b.batch, b.page_size, np.int32))
    second = workloads.scaled(b, kv_indptr=np.array([0] + [int(b.kv_indptr[i + 1]) - h for i, h in enumerate(half)]).cumsum().astype(np.int32),
                              kv_indices=np.concatenate([b.kv_indices[half[i]:b.kv_indptr[i + 1]] for i in range(b.batch)]).astype(np.int32))
    O1, L1 = oracle_full(first)
    O2, L2 = oracle_full(second)
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    out, lse = bsp.merge_state(torch.from_numpy(O1).to(t).cuda(), torch.from_numpy(L1).float().cuda(),
                               torch.from_numpy(O2).to(t).cuda(), torch.from_numpy(L2).float().cuda())
    torch.cuda.synchronize()
    O, L = oracle_full(b)
    compare(out, lse, O, L, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_state_arbitrary_states(bsp, dtype):
    """Arbitrary states with empty ones (LSE = -inf) on either or both sides;
    in-place use into the first operand."""
    rng = np.random.default_rng(31)
    n, H, D = 333, 8, 128
    oa = rng.standard_normal((n, H, D)).astype(np.float32)
    ob = rng.standard_normal((n, H, D)).astype(np.float32)
    la = (rng.standard_normal((n, H)) * 4).astype(np.float32)
    lb = (rng.standard_normal((n, H)) * 4).astype(np.float32)
    la[::7, 0] = -np.inf
    lb[::5, 1] = -np.inf
    la[3, :] = lb[3, :] = -np.inf
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    ta, tb = torch.from_numpy(oa).to(t), torch.from_numpy(ob).to(t)
    Oe, Le = oracle.merge_states(ta.float().numpy(), la, tb.float().numpy(), lb)
    out, lse = bsp.merge_state(ta.cuda(), torch.from_numpy(la).cuda(), tb.cuda(), torch.from_numpy(lb).cuda())
    torch.cuda.synchronize()
    compare(out, lse, Oe, Le, dtype, rounding_aware=True)
    # a pass-through side is copied bit for bit
    pa_rows = np.isneginf(lb) & ~np.isneginf(la)
    assert torch.equal(out.cpu()[torch.from_numpy(pa_rows)], ta[torch.from_numpy(pa_rows)])
    # in place into a
    a_dev, la_dev = ta.cuda(), torch.from_numpy(la).cuda()
    bsp.merge_state(a_dev, la_dev, tb.cuda(), torch.from_numpy(lb).cuda(), out=a_dev, lse_out=la_dev)
    torch.cuda.synchronize()
    assert torch.equal(a_dev, out) and torch.equal(la_dev, lse)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_state_unaligned_rows(bsp, dtype):
    """O arrays that start one element past an aligned address take the
    element-wise path of merge_state; its results equal the vector path's bit
    for bit."""
    rng = np.random.default_rng(32)
    n, H, D = 77, 8, 128
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    oa = torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(t).cuda()
    ob = torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(t).cuda()
    la = torch.from_numpy((rng.standard_normal((n, H)) * 3).astype(np.float32)).cuda()
    lb = torch.from_numpy((rng.standard_normal((n, H)) * 3).astype(np.float32)).cuda()
    ref_o, ref_l = bsp.merge_state(oa, la, ob, lb)

    def shifted(x):
        buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=x.device)
        v = buf[1:].view(x.shape)
        v.copy_(x)
        return v
    ua, ub = shifted(oa), shifted(ob)
    uo = shifted(torch.empty_like(oa))
    assert ua.data_ptr() % 8 != 0
    out, lse = bsp.merge_state(ua, la, ub, lb, out=uo)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_run_rejects_bad_arguments(bsp):
    b = workloads.paged_batch(41, [1, 1], [10, 20], 8, 2, 128, 4, "bf16")
    pa = bsp.PagedAttention("decode", 8, 2, 128, 4, False, torch.bfloat16, max_batch=2, num_ctas=4)
    with pytest.raises(RuntimeError):
        pa.run(*to_dev(b), b.sm_scale)       # no plan yet
    pa.plan(b.kv_indptr, b.last_page_len)
    q, k, v, idx = to_dev(b)
    with pytest.raises(ValueError):
        pa.run(q.float(), k, v, idx)         # wrong dtype
    with pytest.raises(ValueError):
        pa.run(q[:, :4], k, v, idx)          # wrong head count


def test_fused_merge_repeated_runs(bsp):
    """Split decode with the merge inside the kernel: three runs of one plan
    (the arrival counters reset themselves) give identical results that match
    the oracle, and an explicit merge-of-partials launch afterwards changes
    nothing (it recomputes the same fold)."""
    b = workloads.paged_batch(81, [1] * 9, [3000, 17, 900, 4100, 1, 2500, 64, 777, 1500], 32, 8, 128, 16, "bf16",
                              extra_pages=3)
    dev = to_dev(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=37, dev_tensors=dev)
    assert pa.info.num_merges > 0
    q, k, v, idx = dev
    runs = [pa.run(q, k, v, idx, b.sm_scale) for _ in range(3)]
    torch.cuda.synchronize()
    for o2, l2 in runs:
        assert torch.equal(o2, out) and torch.equal(l2, lse)
    O, L = oracle_full(b)
    compare(out, lse, O, L, "bf16")
    o3, l3 = out.clone(), lse.clone()
    pa.run_stages(q, k, v, idx, b.sm_scale, o3, l3)
    N.check(N.load().bsp_run_merge_partials(ctypes.byref(pa.info), ctypes.c_void_p(o3.data_ptr()),
                                            ctypes.c_void_p(l3.data_ptr()), ctypes.c_void_p(pa.workspace.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    assert torch.equal(o3, out) and torch.equal(l3, lse)
    assert pa.check_device_error() == 0


def test_bounded_wait_gives_up(bsp):
    """A wait that nothing completes (the kernels' bounded spin on an mbarrier
    with no arrival) gives up after its limit and records its code in the status
    word, without faulting: the context stays usable and a decode run right
    after it is correct."""
    import time
    from block_sparse_paged_gb300 import _native as N
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    N.check(N.load().bsp_check_bounded_wait(4_000_000, ctypes.c_void_p(status.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == 0x1FF
    assert elapsed < 2.0  # about 2 ms of SM clock, plus launch
    b = workloads.paged_batch(91, [1] * 3, [300, 17, 900], 32, 8, 128, 16, "bf16", extra_pages=2)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=9)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0
