"""Prefill path (tcgen05) and the composable shared-prefix path on the GPU,
through the C ABI, against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare, lib, oracle_full, run_batch, stratified_rows, timed, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    return lib()


CASES = [
    # (seed, qo lens, kv lens, H_qo, H_kv, page, causal, num_ctas)
    (1, [1, 17, 128, 129, 300], [1, 17, 128, 129, 300], 32, 8, 16, True, 152),
    (2, [200, 64, 1000], [200, 64, 1000], 32, 8, 16, True, 7),           # few CTAs, long queues
    (12, [200, 64, 1000], [200, 64, 1000], 32, 8, 16, True, 200),        # splits + merges (48 entries)
    (11, [64, 5, 100], [6000, 700, 3000], 32, 8, 16, True, 40),         # prefix cached: splits + merges
    (3, [33, 5, 260], [100, 5, 900], 8, 8, 8, True, 13),                 # qo < kv (prefix cached)
    (4, [70, 300], [20, 128], 16, 2, 32, True, 5),                       # qo > kv: rows with no key
    (5, [64, 190, 3], [500, 190, 77], 16, 16, 128, False, 9),            # non-causal, g = 1
    (6, [128, 257], [128, 257], 64, 8, 16, True, 3),                     # g = 8
    (7, [1], [0], 32, 8, 16, True, 4),                                   # empty KV
    (8, [65, 300, 17], [65, 300, 17], 32, 8, 1, True, 11),              # page size 1: cp.async gather
    (9, [140, 33], [400, 33], 16, 4, 4, True, 6),                        # page size 4: cp.async gather
    (10, [96, 250], [96, 700], 32, 8, 32, False, 5),                     # page 32 (two pages per box row set)
    (13, [150, 300], [400, 300], 32, 8, 64, True, 9),                    # 64-token pages
    (14, [77, 260], [1000, 260], 16, 4, 256, True, 11),                  # 256-token pages: a page spans two KV tiles
    (15, [100, 0, 77], [300, 50, 77], 32, 2, 16, True, 9),              # g = 16 (16 positions per tile); a request without queries
    (16, [0, 40, 0], [10, 200, 0], 16, 4, 16, False, 4),                 # non-causal; requests without queries or keys
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_random_prefill(bsp, case):
    seed, qo, kv, hq, hk, ps, causal, C = case
    b = workloads.paged_batch(seed, qo, kv, hq, hk, 128, ps, "bf16", causal=causal, extra_pages=2)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=C)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_split_prefill_repeated_runs(bsp):
    """Split prefill (24 reduction-map entries): three runs of one plan give
    identical results that match the oracle, and one more merge-of-partials
    launch afterwards changes nothing (it recomputes the same fold)."""
    import ctypes
    from block_sparse_paged_gb300 import _native as N
    b = workloads.paged_batch(82, [64, 5, 100], [6000, 700, 3000], 32, 8, 128, 16, "bf16", causal=True,
                              extra_pages=2)
    dev = to_dev(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=40, dev_tensors=dev)
    assert pa.info.num_merges > 0
    q, k, v, idx = dev
    runs = [pa.run(q, k, v, idx, b.sm_scale) for _ in range(3)]
    torch.cuda.synchronize()
    for o2, l2 in runs:
        assert torch.equal(o2, out) and torch.equal(l2, lse)
    O, L = oracle_full(b)
    compare(out, lse, O, L, "bf16")
    o3, l3 = out.clone(), lse.clone()
    N.check(N.load().bsp_run_merge_partials(ctypes.byref(pa.info), ctypes.c_void_p(o3.data_ptr()),
                                            ctypes.c_void_p(l3.data_ptr()), ctypes.c_void_p(pa.workspace.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    assert torch.equal(o3, out) and torch.equal(l3, lse)
    assert pa.check_device_error() == 0


def test_prefill_cuda_graph_replay_with_new_plan(bsp):
    """Capture one prefill run (attention kernel + merge of partials), re-plan
    other lengths into the same workspace and replay: the replay matches the
    oracle for the new plan. Both plans split outputs."""
    hq, hk, ps = 32, 8, 16
    a = workloads.paged_batch(61, [64, 5, 100], [6000, 700, 3000], hq, hk, 128, ps, "bf16", causal=True,
                              extra_pages=30)
    bb = workloads.paged_batch(62, [7, 64, 90], [2500, 5200, 90], hq, hk, 128, ps, "bf16", causal=True,
                               extra_pages=30)
    pa = bsp.PagedAttention("prefill", hq, hk, 128, ps, True, torch.bfloat16, max_batch=3, max_qo_tokens=256,
                            num_ctas=40)
    pool = max(a.k_pages.shape[0], bb.k_pages.shape[0])
    n_tok = max(int(a.qo_indptr[-1]), int(bb.qo_indptr[-1]))
    q = torch.zeros((n_tok, hq, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((pool, ps, hk, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    idx = torch.zeros(4096, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")

    def load(batch):
        q[: batch.q.shape[0]].copy_(batch.q)
        k[: batch.k_pages.shape[0]].copy_(batch.k_pages)
        v[: batch.v_pages.shape[0]].copy_(batch.v_pages)
        idx[: len(batch.kv_indices)].copy_(torch.from_numpy(batch.kv_indices))

    load(a)
    pa.plan(a.kv_indptr, a.last_page_len, qo_indptr=a.qo_indptr)
    assert pa.info.num_merges > 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.run(q, k, v, idx, a.sm_scale, out=out, lse=lse)  # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.run(q, k, v, idx, a.sm_scale, out=out, lse=lse)
    for batch in (a, bb):
        if batch is bb:
            load(bb)
            pa.plan(bb.kv_indptr, bb.last_page_len, qo_indptr=bb.qo_indptr)
            assert pa.info.num_merges > 0
        g.replay()
        torch.cuda.synchronize()
        O, L = oracle_full(batch)
        n = int(batch.qo_indptr[-1])
        compare(out[:n], lse[:n], O, L, "bf16")
    assert pa.check_device_error() == 0


def test_ragged_causal_prefill_full_size(bsp):
    """16 requests, qo = kv ~ U{128..2048}, page 16 permuted, 32/8 heads, causal;
    every output row against the oracle; two runs bitwise equal."""
    b = workloads.ragged_causal_prefill_bf16()
    out, lse, pa = run_batch(bsp, b, mode="prefill")
    (O, L), t = timed(oracle_full, b)
    compare(out, lse, O, L, "bf16", oracle_s=t)
    q, k, v, idx = to_dev(b)
    out2, lse2 = pa.run(q, k, v, idx, b.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert pa.check_device_error() == 0
    # the bench's plan: two queues per CTA. No tile is split under either plan,
    # so every output row is computed the same way: bitwise equal
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out3, lse3, pa3 = run_batch(bsp, b, mode="prefill", num_ctas=2 * sms, dev_tensors=(q, k, v, idx))
    assert pa3.info.num_merges == 0 and pa.info.num_merges == 0
    assert torch.equal(out, out3) and torch.equal(lse, lse3)


def test_many_slot_folds_prefill(bsp):
    """A causal prefill planned with many chunks per CTA: the reduce kernel folds
    outputs of 9 to 11 partial states (batches of 8, rescaled to the running
    maximum); against the oracle."""
    b = workloads.paged_batch(62, [700, 130, 1], [3000, 130, 1], 32, 8, 128, 16, "bf16", causal=True,
                              extra_pages=2)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=24, chunks_per_cta=40)
    _, items, merges = pa.plan_arrays()
    assert int(merges["n_slots"].max()) > 8
    n = int(b.qo_indptr[-1])
    compare(out[:n], lse[:n], O, L, "bf16")
    assert pa.check_device_error() == 0


def composable_decode(bsp, sp, num_ctas_prefill=None, num_ctas_decode=None):
    """Prefix view (all queries as one row block over the shared pages, on the
    prefill kernel) and suffix view (decode), merged with merge_state."""
    dev = "cuda"
    q = sp.full.q.to(dev)
    k = sp.full.k_pages.to(dev)
    v = sp.full.v_pages.to(dev)
    pre = bsp.PagedAttention("prefill", 32, 8, 128, sp.full.page_size, False, torch.bfloat16, max_batch=1,
                             max_qo_tokens=sp.prefix.batch * 0 + int(sp.prefix.qo_indptr[-1]),
                             num_ctas=num_ctas_prefill)
    pre.plan(sp.prefix.kv_indptr, sp.prefix.last_page_len, qo_indptr=sp.prefix.qo_indptr)
    suf = bsp.PagedAttention("decode", 32, 8, 128, sp.full.page_size, False, torch.bfloat16,
                             max_batch=sp.suffix.batch, num_ctas=num_ctas_decode)
    suf.plan(sp.suffix.kv_indptr, sp.suffix.last_page_len)
    o1, l1 = pre.run(q, k, v, torch.from_numpy(sp.prefix.kv_indices).to(dev), sp.full.sm_scale)
    o2, l2 = suf.run(q, k, v, torch.from_numpy(sp.suffix.kv_indices).to(dev), sp.full.sm_scale)
    out, lse = bsp.merge_state(o1, l1, o2, l2)
    torch.cuda.synchronize()
    return out, lse


def test_shared_prefix_composable_small(bsp):
    sp = workloads.shared_prefix_decode_bf16(batch=6, prefix_len=512, outlier=700, suffix_lo=1, suffix_hi=90,
                                             seed=51)
    out, lse = composable_decode(bsp, sp, num_ctas_prefill=5, num_ctas_decode=7)
    O, L = oracle_full(sp.full)
    compare(out, lse, O, L, "bf16")


def test_shared_prefix_concurrent_views(bsp):
    """The two views on two streams at once, each on part of the SMs (their plans
    made for those CTA counts), give bit-for-bit the outputs of the same plans
    run one after the other, and those match the oracle."""
    sp = workloads.shared_prefix_decode_bf16(batch=8, prefix_len=1024, outlier=3000, seed=12)
    dev = torch.device("cuda")
    q, k, v = sp.full.q.to(dev), sp.full.k_pages.to(dev), sp.full.v_pages.to(dev)
    ip = torch.from_numpy(sp.prefix.kv_indices).to(dev)
    isf = torch.from_numpy(sp.suffix.kv_indices).to(dev)
    pre = bsp.PagedAttention("prefill", 32, 8, 128, sp.full.page_size, False, torch.bfloat16, max_batch=1,
                             max_qo_tokens=int(sp.prefix.qo_indptr[-1]), num_ctas=50)
    suf = bsp.PagedAttention("decode", 32, 8, 128, sp.full.page_size, False, torch.bfloat16,
                             max_batch=sp.suffix.batch, num_ctas=102)
    pre.plan(sp.prefix.kv_indptr, sp.prefix.last_page_len, qo_indptr=sp.prefix.qo_indptr)
    suf.plan(sp.suffix.kv_indptr, sp.suffix.last_page_len)
    o1, l1 = pre.run(q, k, v, ip, sp.full.sm_scale)
    o2, l2 = suf.run(q, k, v, isf, sp.full.sm_scale)
    ref_o, ref_l = bsp.merge_state(o1, l1, o2, l2)
    torch.cuda.synchronize()
    main, sa, sb = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    c1, c2 = torch.empty_like(o1), torch.empty_like(o2)
    d1, d2 = torch.empty_like(l1), torch.empty_like(l2)
    sa.wait_stream(main)
    sb.wait_stream(main)
    pre.run(q, k, v, ip, sp.full.sm_scale, out=c1, lse=d1, stream=sa)
    suf.run(q, k, v, isf, sp.full.sm_scale, out=c2, lse=d2, stream=sb)
    main.wait_stream(sa)
    main.wait_stream(sb)
    out, lse = bsp.merge_state(c1, d1, c2, d2)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    O, L = oracle_full(sp.full)
    compare(out, lse, O, L, "bf16")


def test_shared_prefix_composable_full_size(bsp):
    """64 requests sharing an 8192-token prefix, suffixes U{64..1024} and one
    32768 outlier: prefix view + suffix view + merge equals attention over the
    full page lists (every output row)."""
    sp = workloads.shared_prefix_decode_bf16()
    out, lse = composable_decode(bsp, sp)
    (O, L), t = timed(oracle_full, sp.full)
    compare(out, lse, O, L, "bf16", oracle_s=t)
    # the bench's split: 32 CTAs for the prefix view (4 equal chunks per tile),
    # the rest for the suffix view
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out2, lse2 = composable_decode(bsp, sp, num_ctas_prefill=32, num_ctas_decode=sms - 32)
    compare(out2, lse2, O, L, "bf16")


def test_vector_sparse_prefill_small(bsp):
    """Page size 1, one 1500-token causal prefill: permuted and contiguous slots
    give bitwise equal outputs (same plan, only the gather differs) and match
    the oracle everywhere."""
    perm, cont = workloads.vector_sparse_prefill_bf16(1500, seed=61)
    o1, l1, _ = run_batch(bsp, perm, mode="prefill", num_ctas=40)
    o2, l2, _ = run_batch(bsp, cont, mode="prefill", num_ctas=40)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O, L = oracle_full(perm)
    compare(o1, l1, O, L, "bf16")


def test_vector_sparse_prefill_full_size(bsp):
    """Page size 1, one 32768-token causal prefill (the long vector-sparse
    prefill) in the bench's configuration (a gather region for the whole page
    table, the default CTA count): a stratified eighth of the rows against the
    oracle (every head, every 8th position with a seeded phase per head, all of
    the first and last query tile; the whole would be ~5 min of fp64 on 16
    cores); permuted == contiguous bitwise, and both equal the cp.async gather
    without a region."""
    perm, cont = workloads.vector_sparse_prefill_bf16()
    n = int(perm.kv_indptr[-1])
    o1, l1, pa = run_batch(bsp, perm, mode="prefill", max_gather_pages=n)
    tok, head = stratified_rows(perm, 8, 23)
    (O, L), t = timed(oracle.attention_rows_of, perm, tok, head)
    compare(o1, l1, O, L, "bf16", rows=(tok, head), oracle_s=t)
    assert pa.check_device_error() == 0
    del pa
    o2, l2, _ = run_batch(bsp, cont, mode="prefill", max_gather_pages=n)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3, _ = run_batch(bsp, perm, mode="prefill")
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


GATHER = [
    # (seed, qo lens, kv lens, H_qo, H_kv, page, causal, num_ctas)
    (131, [65, 300, 17], [65, 300, 17], 32, 8, 1, True, 11),
    (132, [140, 33], [400, 33], 16, 4, 2, True, 6),
    (133, [96, 250, 1], [700, 250, 0], 32, 8, 3, True, 40),      # splits + merges, an empty request
    (134, [200, 90], [900, 90], 32, 8, 12, False, 9),           # 12-token pages (not a power of two)
]


@pytest.mark.parametrize("case", GATHER, ids=[f"gather{c[0]}" for c in GATHER])
def test_gathered_prefill_equals_cp_async(bsp, case):
    """Pages the TMA page gather cannot take (under 8 tokens, or not a power of
    two) with a gather region in the workspace: the page table's pages are
    copied into it in table order and read back by 128-row TMA boxes. Same plan
    and the same shared-memory tiles as the cp.async gather, so the outputs are
    bitwise equal to it; against the oracle. A region one page too small runs
    the cp.async gather."""
    seed, qo, kv, hq, hk, ps, causal, C = case
    b = workloads.paged_batch(seed, qo, kv, hq, hk, 128, ps, "bf16", causal=causal, extra_pages=3)
    n = int(b.kv_indptr[-1])
    dev = to_dev(b)
    o0, l0, _ = run_batch(bsp, b, mode="prefill", num_ctas=C, dev_tensors=dev)
    o1, l1, pa = run_batch(bsp, b, mode="prefill", num_ctas=C, dev_tensors=dev, max_gather_pages=n)
    assert pa.info.off_gather > 0 and pa.info.num_table_pages == n
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert pa.check_device_error() == 0
    O, L = oracle_full(b)
    compare(o1, l1, O, L, "bf16")
    o2, l2, _ = run_batch(bsp, b, mode="prefill", num_ctas=C, dev_tensors=dev, max_gather_pages=max(1, n - 1))
    assert torch.equal(o0, o2) and torch.equal(l0, l2)


def test_gathered_prefill_variants_and_sink(bsp):
    """The gathered path with a sliding window, a soft-cap and sinks (the
    variant kernel), page size 1; against the oracle."""
    b = workloads.paged_batch(135, [200, 90], [700, 90], 16, 4, 128, 1, "bf16", causal=True, extra_pages=2)
    b.window_left, b.soft_cap = 77, 2.5
    sk = np.random.default_rng(135).uniform(-2.0, 4.0, size=16)
    O, L = oracle_full(b, sink=sk)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=7, sink=sk, max_gather_pages=int(b.kv_indptr[-1]))
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_equal_share_prefill(bsp):
    """Causal ragged prefill under the equal-share schedule (tiles split across
    CTAs at page boundaries, merged by the reduce kernel); against the oracle."""
    b = workloads.paged_batch(137, [300, 65, 1000, 1], [300, 65, 1000, 0], 32, 8, 128, 16, "bf16", causal=True,
                              extra_pages=2)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=23, schedule="equal")
    assert pa.info.num_merges > 0
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_gather_reports_page_ids_out_of_range(bsp):
    """The gather checks every page id against the pool size: an id outside it
    gives a zero page and the status word 0x301 (no out-of-range read)."""
    b = workloads.paged_batch(136, [50, 40], [50, 40], 32, 8, 128, 1, "bf16", causal=True, extra_pages=2)
    q, k, v, idx = to_dev(b)
    idx[3] = k.shape[0] + 5
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=4, dev_tensors=(q, k, v, idx),
                             max_gather_pages=int(b.kv_indptr[-1]))
    assert pa.check_device_error() == 0x301
    assert pa.check_device_error() == 0
