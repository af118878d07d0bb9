"""The oracle planner against the pages' worked example and the invariants
the scheduling argument fixes, plus planted mistakes it must catch (CPU)."""
import importlib.util
import itertools
import math
import sys

import numpy as np
import pytest

from conftest import golden
from oracle import plan as oplan



def pin_lpt_worked_example(pl):
    """Overview ⑨: KV [1000,100,100,50], 4 CTAs, cost = KV length."""
    g = golden("lpt_worked_example.json")
    names = "ABCD"
    p = pl.plan([1] * 4, g["kv_lens"], 1, 1, 1, g["num_ctas"], 1, False, alpha=g["alpha"], beta=g["beta"])
    pr = g["printed"]
    assert p.total_work == pr["total_work"] and p.chunk_len == pr["chunk_len"], (p.total_work, p.chunk_len)
    got = [[[names[it.b], it.kv_end - it.kv_start] for it in q] for q in p.queues]
    assert got == pr["cta_queues_as_request_and_length"], got
    assert p.cta_cost[3] == pr["cta3_total"]
    a_chunks = sorted([it for q in p.queues for it in q if it.b == 0], key=lambda it: it.kv_start)
    assert [it.kv_end - it.kv_start for it in a_chunks] == pr["chunks_of_A"]
    # the cost model of the source (2 qo_len + kv_len) leaves this assignment unchanged
    p2 = pl.plan([1] * 4, g["kv_lens"], 1, 1, 1, g["num_ctas"], 1, False)
    assert [[(it.b, it.kv_start, it.kv_end) for it in q] for q in p2.queues] == \
           [[(it.b, it.kv_start, it.kv_end) for it in q] for q in p.queues]


def pin_capacity_formula(pl):
    """Technical review eq 13: 2 C T_q H_q (d + 1) = 13,209,600 for C=100, T_q=16, H_q=32, d=128."""
    g = golden("partial_capacity.json")
    e = pl.partial_capacity_elements(g["C"], g["T_q"], g["H_q"], g["d"])
    assert e == g["printed"]["elements"]
    assert round(e * 4 / 2**20, 1) == g["printed"]["mib_at_4_bytes"]


def _cases():
    rng = np.random.default_rng(7)
    cases = []
    for i in range(40):
        B = int(rng.integers(1, 9))
        causal = bool(i % 2)
        decode = i % 3 == 0
        g = int(rng.choice([1, 2, 4]))
        kv = rng.integers(0, 300, size=B)
        qo = np.ones(B, int) if decode else np.minimum(kv, rng.integers(1, 60, size=B)) if causal else rng.integers(1, 60, size=B)
        qo = np.maximum(qo, 1)
        tile = g if decode else int(rng.choice([16, 32])) * g
        cases.append(dict(qo=qo.tolist(), kv=kv.tolist(), hk=int(rng.integers(1, 4)), g=g, tile=tile,
                          C=int(rng.integers(1, 20)), ps=int(rng.choice([1, 4, 16])), causal=causal))
    return cases


def pin_coverage(pl):
    """Every (request, kv head, query position, visible KV position) is covered
    exactly once, and each multi-chunk output's slots are consecutive and in
    ascending chunk order (walkthrough §VIII.5 reduction map)."""
    for c in _cases():
        p = pl.plan(c["qo"], c["kv"], c["hk"], c["g"], c["tile"], c["C"], c["ps"], c["causal"])
        items = [it for q in p.queues for it in q]
        by_out = {}
        for it in items:
            by_out.setdefault((it.b, it.tile, it.kv_head), []).append(it)
        for b in range(len(c["qo"])):
            ntile = -(-c["qo"][b] * c["g"] // c["tile"])
            for t in range(ntile):
                per = c["tile"] // c["g"]
                last_pos = min(c["qo"][b], (t + 1) * per) - 1
                vis = c["kv"][b] if not c["causal"] else max(0, min(c["kv"][b], last_pos + c["kv"][b] - c["qo"][b] + 1))
                for h in range(c["hk"]):
                    chunks = sorted(by_out.pop((b, t, h)), key=lambda it: it.kv_start)
                    covered = [x for it in chunks for x in range(it.kv_start, it.kv_end)]
                    assert covered == list(range(vis)), (c, b, t, h)
                    assert all(it.kv_end - it.kv_start <= p.chunk_len for it in chunks)
                    assert all(it.kv_start % c["ps"] == 0 for it in chunks)
                    if len(chunks) == 1:
                        assert chunks[0].slot == -1
                    else:
                        slots = [it.slot for it in chunks]
                        assert slots == list(range(slots[0], slots[0] + len(chunks)))
        assert not by_out
        # reduction map: outputs in (b, tile, kv_head) order with consecutive slot ranges
        nxt = 0
        for o in p.outputs:
            assert o.slot_begin == nxt and o.n_slots >= 2
            nxt += o.n_slots
        assert nxt == p.num_partials


def pin_chunk_len_and_bounds(pl):
    """L = max(1, ceil(W / C)) rounded up to a page (technical review Algorithm 2
    step 4); partial slots stay within 2 C (eq 13's factor of two, per tile and
    kv head); the makespan is at least eq 12's bound."""
    for c in _cases():
        p = pl.plan(c["qo"], c["kv"], c["hk"], c["g"], c["tile"], c["C"], c["ps"], c["causal"])
        W = sum(-(-q * c["g"] // c["tile"]) * k * c["hk"] for q, k in zip(c["qo"], c["kv"]))
        assert p.total_work == W
        L = max(1, math.ceil(W / c["C"]))
        assert p.chunk_len == math.ceil(L / c["ps"]) * c["ps"]
        assert p.num_partials <= 2 * c["C"]
        costs = []
        for q in p.queues:
            for it in q:
                lq = min(c["qo"][it.b], (it.tile + 1) * (c["tile"] // c["g"])) - it.tile * (c["tile"] // c["g"])
                costs.append(2 * lq + (it.kv_end - it.kv_start))
        assert max(p.cta_cost) >= pl.makespan_lower_bound(costs, c["C"]) - 1e-9
        assert sum(p.cta_cost) == sum(costs)


def pin_lpt_quality(pl):
    """Longest-first greedy: each queue is in non-increasing chunk length order,
    and the makespan is within Graham's (4/3 - 1/(3C)) of the optimum, checked
    by brute force over every assignment of up to 8 chunks to up to 3 CTAs."""
    rng = np.random.default_rng(8)
    for _ in range(60):
        B = int(rng.integers(1, 9))
        C = int(rng.integers(1, 4))
        kv = rng.integers(1, 50, size=B).tolist()
        p = pl.plan([1] * B, kv, 1, 1, 1, C, 1, False, alpha=0, beta=1)
        for q in p.queues:
            lens = [it.kv_end - it.kv_start for it in q]
            assert lens == sorted(lens, reverse=True)
        sizes = [it.kv_end - it.kv_start for q in p.queues for it in q]
        if len(sizes) > 8:
            continue
        best = min(max(sum(s for s, a in zip(sizes, asg) if a == c) for c in range(C))
                   for asg in itertools.product(range(C), repeat=len(sizes)))
        assert max(p.cta_cost) <= (4 / 3 - 1 / (3 * C)) * best + 1e-9, (sizes, C, p.cta_cost, best)


def pin_determinism(pl):
    c = _cases()[5]
    a = pl.plan(c["qo"], c["kv"], c["hk"], c["g"], c["tile"], c["C"], c["ps"], c["causal"])
    b = pl.plan(c["qo"], c["kv"], c["hk"], c["g"], c["tile"], c["C"], c["ps"], c["causal"])
    assert a.queues == b.queues and a.outputs == b.outputs


def pin_empty_tiles(pl):
    """A request with no KV still gets one empty chunk per (tile, kv head)."""
    p = pl.plan([1, 1], [0, 5], 2, 1, 1, 3, 4, False)
    items = [it for q in p.queues for it in q]
    assert sorted((it.b, it.kv_head, it.kv_start, it.kv_end) for it in items if it.b == 0) == [(0, 0, 0, 0), (0, 1, 0, 0)]


def pin_chunks_per_cta(pl):
    """s chunks per CTA: L = ceil(W / (s C)). Two 4096-token tiles on 2 CTAs
    with s = 4 give L = 1024, four equal chunks per tile and four chunks (4096
    tokens plus alpha per chunk) per CTA; s = 1 (and 0, read as 1) keeps the
    pages' L = ceil(W / C) = 4096, one chunk per tile."""
    p = pl.plan([1, 1], [4096, 4096], 1, 1, 1, 2, 1, False, alpha=2, beta=1, chunks_per_cta=4)
    assert p.chunk_len == 1024 and p.num_partials == 8
    assert sorted(len(q) for q in p.queues) == [4, 4] and p.cta_cost == [4096 + 8, 4096 + 8]
    for s in (0, 1):
        p1 = pl.plan([1, 1], [4096, 4096], 1, 1, 1, 2, 1, False, chunks_per_cta=s)
        assert p1.chunk_len == 4096 and p1.num_partials == 0
    p3 = pl.plan([1], [1000], 1, 1, 1, 1, 16, False, chunks_per_cta=3)  # ceil(1000 / 3) = 334 -> 336 (pages)
    assert p3.chunk_len == 336 and [(it.kv_start, it.kv_end) for it in p3.queues[0]] == [(0, 336), (336, 672), (672, 1000)]


def pin_traffic_ratio(pl):
    """Technical review eq 15 limits: n = 1 gives 1; no suffix gives n."""
    assert pl.prefix_traffic_ratio(1, 8192, 300) == pytest.approx(1.0)
    assert pl.prefix_traffic_ratio(64, 8192, 0) == pytest.approx(64.0)


def pin_equal_share_example(pl):
    """Equal shares (this build's extension) on a case worked out by hand from
    the definition: two 10-token decode requests, one kv head, 3 CTAs. V = 20,
    cuts floor(20/3) = 6 and floor(40/3) = 13. Page size 1: CTA 0 takes [0, 6)
    of request 0, CTA 1 its [6, 10) and [0, 3) of request 1, CTA 2 [3, 10);
    both requests split in two (slots 0, 1 and 2, 3). Page size 4: cut 6 moves
    down to key 4, cut 13 (key 3 of request 1) down to key 0, the start of
    request 1: [0, 4) | [4, 10) | request 1 whole."""
    p = pl.plan([1, 1], [10, 10], 1, 1, 1, 3, 1, False, schedule="equal")
    got = [[(it.b, it.kv_start, it.kv_end, it.slot) for it in q] for q in p.queues]
    assert got == [[(0, 0, 6, 0)], [(0, 6, 10, 1), (1, 0, 3, 2)], [(1, 3, 10, 3)]], got
    assert [(o.b, o.slot_begin, o.n_slots) for o in p.outputs] == [(0, 0, 2), (1, 2, 2)]
    p = pl.plan([1, 1], [10, 10], 1, 1, 1, 3, 4, False, schedule="equal")
    got = [[(it.b, it.kv_start, it.kv_end, it.slot) for it in q] for q in p.queues]
    assert got == [[(0, 0, 4, 0)], [(0, 4, 10, 1)], [(1, 0, 10, -1)]], got
    assert p.chunk_len == 10 and p.num_partials == 2


def pin_equal_share_balance(pl):
    """Equal shares: every (request, kv head, visible position) exactly once; each
    CTA's KV within a page of V / C (ceil(V / C) + page_size - 1 at most, floor(V / C)
    - (page_size - 1) at least, for shares that do not end at a tile's end);
    queues in the order of the concatenation; at most tiles + C - 1 chunks."""
    for c in _cases():
        p = pl.plan(c["qo"], c["kv"], c["hk"], c["g"], c["tile"], c["C"], c["ps"], c["causal"], schedule="equal")
        order = []  # (b, tile, kv_head) in concatenation order with their visible lengths
        for b in range(len(c["qo"])):
            ntile = -(-c["qo"][b] * c["g"] // c["tile"])
            for t in range(ntile):
                per = c["tile"] // c["g"]
                last_pos = min(c["qo"][b], (t + 1) * per) - 1
                vis = c["kv"][b] if not c["causal"] else max(0, min(c["kv"][b], last_pos + c["kv"][b] - c["qo"][b] + 1))
                for h in range(c["hk"]):
                    order.append(((b, t, h), vis))
        V = sum(v for _, v in order)
        pos = {}
        acc = 0
        for key, v in order:
            pos[key] = acc
            acc += v
        items = [it for q in p.queues for it in q]
        assert len(items) <= len(order) + c["C"] - 1
        cover = {}
        for it in items:
            cover.setdefault((it.b, it.tile, it.kv_head), []).extend(range(it.kv_start, it.kv_end))
        assert set(cover) == {key for key, _ in order}  # every tile has a chunk, empty tiles one empty chunk
        for key, v in order:
            assert sorted(cover[key]) == list(range(v)), (c, key)
        for ci, q in enumerate(p.queues):
            load = sum(it.kv_end - it.kv_start for it in q)
            assert load <= -(-V // c["C"]) + c["ps"] - 1, (c, ci, load)
            starts = [pos[(it.b, it.tile, it.kv_head)] + it.kv_start for it in q if it.kv_end > it.kv_start]
            assert starts == sorted(starts)


ALL_PLAN_PINS = [pin_lpt_worked_example, pin_capacity_formula, pin_coverage, pin_chunk_len_and_bounds,
                 pin_lpt_quality, pin_determinism, pin_empty_tiles, pin_chunks_per_cta, pin_traffic_ratio,
                 pin_equal_share_example, pin_equal_share_balance]


@pytest.mark.parametrize("pin", ALL_PLAN_PINS, ids=lambda f: f.__name__)
def test_plan_pin(pin):
    pin(oplan)


PLAN_MUTATIONS = [
    ("floor_chunk", "L = max(1, -(-W // (num_ctas * max(1, chunks_per_cta))))",
     "L = max(1, W // (num_ctas * max(1, chunks_per_cta)))"),
    ("chunks_per_cta_ignored", "L = max(1, -(-W // (num_ctas * max(1, chunks_per_cta))))",
     "L = max(1, -(-W // num_ctas))"),
    ("no_page_rounding", "L = -(-L // page_size) * page_size", "L = L"),
    ("shortest_first", "chunks.sort(key=lambda c: (-(c[4] - c[3]), c[0], c[1], c[2], c[3]))",
     "chunks.sort(key=lambda c: ((c[4] - c[3]), c[0], c[1], c[2], c[3]))"),
    ("heap_sign_flipped", "heapq.heappush(heap, (cost + alpha * lq + beta * (e - s), cta))",
     "heapq.heappush(heap, (cost - alpha * lq - beta * (e - s), cta))"),
    ("causal_top_left", "return max(0, min(kv_len, last_pos + kv_len - qo_len + 1))",
     "return max(0, min(kv_len, last_pos + 1))"),
    ("no_head_factor", "W += kv_lens[b]", "W += kv_lens[b] if h == 0 else 0"),
    ("no_empty_chunk", "or [(0, 0)]", "or []"),
    ("slots_not_consecutive", "chunks.append((b, t, h, s, e, lq, next_slot + i))",
     "chunks.append((b, t, h, s, e, lq, next_slot + 2 * i))"),
    ("equal_cuts_rounded_up", "cuts = [c * V // num_ctas for c in range(num_ctas + 1)]",
     "cuts = [-(-c * V // num_ctas) for c in range(num_ctas + 1)]"),
    ("equal_cuts_not_on_pages", "cuts[c] = P + (key // page_size * page_size - lo)", "cuts[c] = P + (key - lo)"),
    ("equal_empty_tile_dropped", "queues[owner].append(Item(b, t, h, 0, 0, -1))", "pass"),
    ("equal_slots_shared", "queues[c].append(Item(b, t, h, s, e, next_slot + k if len(pieces) > 1 else -1))",
     "queues[c].append(Item(b, t, h, s, e, next_slot if len(pieces) > 1 else -1))"),
]


@pytest.mark.parametrize("name,old,new", PLAN_MUTATIONS, ids=[m[0] for m in PLAN_MUTATIONS])
def test_plan_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(oplan.__file__).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"plan_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"plan_mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    caught = []
    for pin in ALL_PLAN_PINS:
        try:
            pin(mod)
        except Exception:
            caught.append(pin.__name__)
    assert caught, name
