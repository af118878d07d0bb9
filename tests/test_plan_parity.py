"""The library's C++ planner against the oracle planner: bit-exact queues,
items and reduction map on the same lengths (host only, no device)."""
import numpy as np
import pytest

import workloads
from oracle import plan as oplan


@pytest.fixture(scope="module")
def bsp():
    from block_sparse_paged_gb300 import build
    build.build()
    import block_sparse_paged_gb300 as bsp
    return bsp


def run_both(bsp, mode, qo_lens, kv_lens, page_size, H_qo, H_kv, causal, C, alpha=2, beta=1, D=128,
             max_batch=None, max_qo=None, window_left=-1, s=1, schedule="lpt"):
    qo_lens = np.asarray(qo_lens, np.int64)
    kv_lens = np.asarray(kv_lens, np.int64)
    B = len(kv_lens)
    npages = np.array([-(-int(k) // page_size) for k in kv_lens], np.int64)
    last = np.array([int(k) - (n - 1) * page_size if n > 0 else 0 for k, n in zip(kv_lens, npages)], np.int32)
    kv_indptr = np.zeros(B + 1, np.int32)
    kv_indptr[1:] = np.cumsum(npages)
    qo_indptr = np.zeros(B + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    g = H_qo // H_kv
    prob = bsp.make_problem(mode, H_qo, H_kv, D, page_size, causal, __import__("torch").bfloat16,
                            window_left=window_left)
    sched = bsp._native.BSP_SCHEDULE_EQUAL_SHARES if schedule == "equal" else bsp._native.BSP_SCHEDULE_LPT
    cap = bsp.Capacity(max_batch or B, C, max_qo or int(qo_indptr[-1]), s, 0, sched)
    info, queue, items, merges = bsp.plan_host(prob, cap, kv_indptr, last,
                                               None if mode == bsp.BSP_MODE_DECODE and np.all(qo_lens == 1) else qo_indptr,
                                               alpha, beta)
    tile = g if mode == bsp.BSP_MODE_DECODE else 256
    ref = oplan.plan(qo_lens.tolist(), kv_lens.tolist(), H_kv, g, tile, C, page_size, causal, alpha, beta,
                     window_left=window_left, chunks_per_cta=s, schedule=schedule)
    return info, queue, items, merges, ref, qo_indptr, kv_indptr


def assert_same(info, queue, items, merges, ref, qo_indptr, kv_indptr):
    assert info.chunk_len == ref.chunk_len and info.total_work == ref.total_work
    assert info.num_partials == ref.num_partials
    got = [[(int(it["b"]), int(it["tile"]), int(it["kv_head"]), int(it["kv_start"]), int(it["kv_end"]), int(it["slot"]))
            for it in items[queue[c]:queue[c + 1]]] for c in range(len(queue) - 1)]
    want = [[(it.b, it.tile, it.kv_head, it.kv_start, it.kv_end, it.slot) for it in q] for q in ref.queues]
    assert got == want
    got_m = [(int(m["b"]), int(m["tile"]), int(m["kv_head"]), int(m["slot_begin"]), int(m["n_slots"])) for m in merges]
    want_m = [(o.b, o.tile, o.kv_head, o.slot_begin, o.n_slots) for o in ref.outputs]
    assert got_m == want_m
    # derived fields the kernels read
    per = info.tile_rows // info.group
    for it in items:
        b = int(it["b"])
        assert it["pos0"] == it["tile"] * per
        assert it["q_tok0"] == qo_indptr[b] + it["pos0"]
        assert it["qo_len"] == qo_indptr[b + 1] - qo_indptr[b]
        assert it["page_base"] == kv_indptr[b]
        assert it["n_pos"] == min(int(it["qo_len"]), int(it["pos0"]) + per) - it["pos0"]
        if it["slot"] < 0:
            assert it["merge"] == -1
        else:  # the reduction-map entry whose slot range holds the item's slot
            m = merges[int(it["merge"])]
            assert m["slot_begin"] <= it["slot"] < m["slot_begin"] + m["n_slots"]
            assert (m["b"], m["tile"], m["kv_head"]) == (it["b"], it["tile"], it["kv_head"])
    assert all(int(m["arrived"]) == 0 for m in merges)


def test_lpt_worked_example(bsp):
    out = run_both(bsp, bsp.BSP_MODE_DECODE, [1] * 4, [1000, 100, 100, 50], 1, 1, 1, False, 4, alpha=0, beta=1)
    assert_same(*out)
    q, items = out[1], out[2]
    assert [int(items[i]["kv_end"] - items[i]["kv_start"]) for i in range(q[3], q[4])] == [100, 100, 61, 50]


@pytest.mark.parametrize("seed", range(30))
def test_random_decode_and_prefill(bsp, seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 40))
    H_kv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    ps = int(rng.choice([1, 3, 16, 64]))
    C = int(rng.integers(1, 400))
    kv = rng.integers(0, 5000, size=B)
    if seed % 2 == 0:
        out = run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(B, int), kv, ps, H_kv * g, H_kv, bool(seed % 4 == 0), C)
    else:
        causal = bool(seed % 3)
        qo = np.maximum(1, np.minimum(kv, rng.integers(1, 700, size=B))) if causal else rng.integers(1, 700, size=B)
        out = run_both(bsp, bsp.BSP_MODE_PREFILL, qo, kv, ps, H_kv * g, H_kv, causal, C)
    assert_same(*out)


@pytest.mark.parametrize("seed", range(12))
def test_random_plans_with_chunks_per_cta(bsp, seed):
    # s > 1: L = ceil(W / (s C)); the capacity bounds (tiles + s C items, 2 s C
    # partial slots) must hold for every s, so the random cases reach s = 64
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 40))
    H_kv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 4, 8]))
    ps = int(rng.choice([1, 3, 16]))
    C = int(rng.integers(1, 200))
    s = int(rng.choice([2, 4, 7, 64]))
    kv = rng.integers(0, 5000, size=B)
    if seed % 2 == 0:
        out = run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(B, int), kv, ps, H_kv * g, H_kv, False, C, alpha=64, s=s)
    else:
        qo = np.maximum(1, np.minimum(kv, rng.integers(1, 700, size=B)))
        out = run_both(bsp, bsp.BSP_MODE_PREFILL, qo, kv, ps, H_kv * g, H_kv, True, C, s=s)
    assert_same(*out)
    info, queue = out[0], out[1]
    assert info.num_items <= info.cap_items and info.num_partials <= info.cap_partials


def test_vector_sparse_decode_balance_with_chunks_per_cta(bsp):
    # 32 requests x 4096 tokens x 8 kv heads on 152 queues: with s = 1 no tile is
    # split (L = 6899) and 104 queues carry two tiles while 48 carry one; s = 4
    # splits every tile so that the busiest queue carries at most 0.92 / 0.83 of
    # the s = 1 load
    loads = {}
    for s in (1, 4):
        out = run_both(bsp, bsp.BSP_MODE_DECODE, [1] * 32, [4096] * 32, 1, 64, 8, False, 152, alpha=64, s=s)
        assert_same(*out)
        loads[s] = max(out[4].cta_cost)
    ideal = 32 * 4096 * 8 / 152
    assert ideal / loads[1] < 0.84 and ideal / loads[4] > 0.91


def test_benchmark_workload_lengths(bsp):
    _, kv2 = workloads.batched_decode_lengths()
    assert_same(*run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(64, int), kv2, 16, 32, 8, False, 304))
    _, l4 = workloads.ragged_causal_prefill_lengths()
    assert_same(*run_both(bsp, bsp.BSP_MODE_PREFILL, l4, l4, 16, 32, 8, True, 152))
    _, suf = workloads.shared_prefix_suffix_lengths()
    assert_same(*run_both(bsp, bsp.BSP_MODE_PREFILL, [64], [8192], 16, 32, 8, False, 152))
    assert_same(*run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(64, int), suf, 16, 32, 8, False, 304))


def test_capacity_and_metadata_errors(bsp):
    import torch
    prob = bsp.make_problem(bsp.BSP_MODE_DECODE, 8, 2, 128, 4, False, torch.bfloat16)
    with pytest.raises(bsp.BspError, match="CAPACITY"):
        bsp.plan_host(prob, bsp.Capacity(2, 8, 2), [0, 1, 2, 3], [1, 1, 1])          # batch 3 > 2
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_host(prob, bsp.Capacity(4, 8, 4), [0, 2, 1], [1, 1])                # indptr decreasing
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_host(prob, bsp.Capacity(4, 8, 4, 65), [0, 1, 2], [1, 1])            # chunks_per_cta > 64
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_host(prob, bsp.Capacity(4, 8, 4, -1), [0, 1, 2], [1, 1])
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_host(prob, bsp.Capacity(4, 8, 4), [0, 2, 3], [1, 5])                # last_page_len > page
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_host(prob, bsp.Capacity(4, 8, 4), [0, 2, 3], [0, 1])                # last_page_len 0
    pre = bsp.make_problem(bsp.BSP_MODE_PREFILL, 8, 2, 128, 16, True, torch.bfloat16)
    with pytest.raises(bsp.BspError, match="CAPACITY"):
        bsp.plan_host(pre, bsp.Capacity(4, 8, 10), [0, 1, 2], [16, 16], qo_indptr=[0, 6, 12])  # 12 > 10 tokens
    bad = bsp.make_problem(bsp.BSP_MODE_PREFILL, 6, 2, 128, 16, True, torch.bfloat16)   # 128 % 3 != 0
    with pytest.raises(bsp.BspError, match="128 %"):
        bsp.plan_host(bad, bsp.Capacity(4, 8, 10), [0, 1], [16], qo_indptr=[0, 6])


def test_partials_within_eq13_bound(bsp):
    rng = np.random.default_rng(5)
    for _ in range(20):
        B = int(rng.integers(1, 30))
        C = int(rng.integers(1, 64))
        kv = rng.integers(1, 20000, size=B)
        info, *_ = run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(B, int), kv, 16, 32, 8, False, C)
        assert info.num_partials <= 2 * C <= info.cap_partials
        assert info.num_items <= info.cap_items and info.num_merges <= info.cap_merges


@pytest.mark.parametrize("case", [
    # (mode, qo lens, kv lens, page, H_qo, H_kv, causal, C, window_left)
    ("decode", [1] * 6, [900, 30, 2000, 1, 513, 64], 16, 32, 8, False, 13, 100),
    ("decode", [1] * 4, [40, 300, 7, 1000], 1, 8, 8, False, 5, 33),
    ("prefill", [300, 65, 1200], [300, 65, 1500], 16, 32, 8, True, 11, 200),
    ("prefill", [700, 90], [700, 400], 8, 16, 4, True, 7, 64),
    ("prefill", [128, 40], [500, 40], 4, 8, 8, False, 9, 17),
])
def test_window_plan_parity_and_coverage(bsp, case):
    """Sliding window: the C planner equals the oracle planner bit for bit, and
    the chunks of every output tile cover each of its rows' visible keys
    (j <= i + kv_len - qo_len when causal, j >= i + kv_len - qo_len - w) once."""
    mode_s, qo, kv, ps, hq, hk, causal, C, w = case
    mode = bsp.BSP_MODE_DECODE if mode_s == "decode" else bsp.BSP_MODE_PREFILL
    info, queue, items, merges, ref, qo_indptr, kv_indptr = run_both(bsp, mode, qo, kv, ps, hq, hk, causal, C,
                                                                    window_left=w)
    assert_same(info, queue, items, merges, ref, qo_indptr, kv_indptr)
    per = info.tile_rows // info.group
    covered = {}
    for it in items:
        key = (int(it["b"]), int(it["tile"]), int(it["kv_head"]))
        covered.setdefault(key, []).append((int(it["kv_start"]), int(it["kv_end"])))
    for (b, t, h), ranges in covered.items():
        ranges.sort()
        for (s0, e0), (s1, e1) in zip(ranges, ranges[1:]):
            assert e0 == s1  # contiguous, no overlap
        lo, hi = ranges[0][0], ranges[-1][1]
        for p in range(t * per, min(qo[b], (t + 1) * per)):
            vis_hi = min(kv[b], p + kv[b] - qo[b] + 1) if causal else kv[b]
            vis_lo = max(0, p + kv[b] - qo[b] - w)
            if vis_hi > vis_lo:
                assert lo <= vis_lo and vis_hi <= hi, (b, t, p, lo, hi, vis_lo, vis_hi)
                assert lo % ps == 0


@pytest.mark.parametrize("seed", range(24))
def test_random_equal_share_plans(bsp, seed):
    """The equal-share schedule: C++ and oracle planners bit-exact on random
    decode and prefill batches (windows and empty requests included), within
    the s = 1 capacity bounds."""
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 40))
    H_kv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    ps = int(rng.choice([1, 3, 16, 64]))
    C = int(rng.integers(1, 400))
    kv = rng.integers(0, 5000, size=B)
    kv[rng.random(B) < 0.1] = 0
    w = int(rng.choice([-1, 300])) if seed % 3 == 0 else -1
    if seed % 2 == 0:
        out = run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(B, int), kv, ps, H_kv * g, H_kv, False, C, alpha=64,
                       window_left=w, schedule="equal")
    else:
        causal = bool(seed % 3)
        qo = np.maximum(1, np.minimum(np.maximum(kv, 1), rng.integers(1, 700, size=B))) if causal else rng.integers(1, 700, size=B)
        out = run_both(bsp, bsp.BSP_MODE_PREFILL, qo, kv, ps, H_kv * g, H_kv, causal, C, window_left=w,
                       schedule="equal")
    assert_same(*out)
    info = out[0]
    assert info.num_items <= info.cap_items and info.num_partials <= info.cap_partials


def test_equal_share_benchmark_workloads(bsp):
    """The page-size-1 decode (32 x 4096 tokens, 8 kv heads) on 152 CTAs: every CTA
    gets 6898 or 6899 tokens in at most 3 items; and the other decode workloads."""
    out = run_both(bsp, bsp.BSP_MODE_DECODE, [1] * 32, [4096] * 32, 1, 64, 8, False, 152, alpha=64,
                   schedule="equal")
    assert_same(*out)
    ref = out[4]
    loads = [sum(it.kv_end - it.kv_start for it in q) for q in ref.queues]
    assert set(loads) <= {6898, 6899}
    assert max(len(q) for q in ref.queues) <= 3
    _, kv2 = workloads.batched_decode_lengths()
    assert_same(*run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(64, int), kv2, 16, 32, 8, False, 152, alpha=64,
                          schedule="equal"))
    _, suf = workloads.shared_prefix_suffix_lengths()
    assert_same(*run_both(bsp, bsp.BSP_MODE_DECODE, np.ones(64, int), suf, 16, 32, 8, False, 120, alpha=64,
                          schedule="equal"))
