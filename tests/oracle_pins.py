"""Pins for the C oracle: checks against what the pages print and what the
mathematics fixes, written as functions of an oracle instance so that the same
checks can be run against deliberately broken copies of the oracle.

Each pin names the passage (page title and section) it comes from.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import logsumexp, softmax

from conftest import golden
import workloads

# ---------------------------------------------------------------------------
# tiny hand-built batches
# ---------------------------------------------------------------------------


def one_request(keys, values, q, page_size=None, sm_scale=1.0, order=None):
    """A single decode request over len(keys) tokens, pages laid out in `order`."""
    keys = np.asarray(keys, np.float32)
    values = np.asarray(values, np.float32)
    n, D = keys.shape
    ps = page_size or n
    npages = -(-n // ps)
    order = list(range(npages)) if order is None else list(order)
    pool = max(order) + 1
    k = np.full((pool, ps, 1, D), np.nan, np.float32)
    v = np.full((pool, ps, 1, D), np.nan, np.float32)
    for t in range(n):
        k[order[t // ps], t % ps, 0] = keys[t]
        v[order[t // ps], t % ps, 0] = values[t]
    last = n - (npages - 1) * ps
    return dict(q=np.asarray(q, np.float32).reshape(1, 1, D), k_pages=k, v_pages=v,
                qo_indptr=[0, 1], kv_indptr=[0, npages], kv_indices=order, last_page_len=[last],
                num_qo_heads=1, num_kv_heads=1, page_size=ps, causal=False, sm_scale=sm_scale)


def run(orc, case):
    o, lse = orc.attention(**case)
    return o[0, 0], lse[0, 0]


def dense_reference(batch: workloads.PagedBatch):
    """Library-routine attention on a CONTIGUOUS batch (pages in request order).

    The logical KV of request b is a plain slice of the flattened pool; query
    head h reads the h-th entry of the kv-head axis repeated g times; the
    bottom-right causal mask is numpy's tril with offset kv_len - qo_len, the
    sliding window numpy's triu with offset kv_len - qo_len - window_left, the
    soft-cap numpy's tanh on the scaled scores; the softmax and log-sum-exp are
    scipy's."""
    assert np.array_equal(batch.kv_indices, np.arange(len(batch.kv_indices)))
    kf = batch.k_pages.float().numpy().reshape(-1, batch.num_kv_heads, batch.head_dim)
    vf = batch.v_pages.float().numpy().reshape(-1, batch.num_kv_heads, batch.head_dim)
    qf = batch.q.float().numpy().astype(np.float64)
    g = batch.num_qo_heads // batch.num_kv_heads
    n_tok = int(batch.qo_indptr[-1])
    O = np.zeros((n_tok, batch.num_qo_heads, batch.head_dim))
    L = np.full((n_tok, batch.num_qo_heads), -np.inf)
    for b in range(batch.batch):
        q0, q1 = int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])
        t0 = int(batch.kv_indptr[b]) * batch.page_size
        kvl = int(batch.kv_lens[b])
        K = np.repeat(kf[t0:t0 + kvl].astype(np.float64), g, axis=1)   # [kvl, H_qo, D]
        V = np.repeat(vf[t0:t0 + kvl].astype(np.float64), g, axis=1)
        for h in range(batch.num_qo_heads):
            S = batch.sm_scale * qf[q0:q1, h] @ K[:, h].T               # [qo, kvl]
            if batch.soft_cap > 0:
                S = batch.soft_cap * np.tanh(S / batch.soft_cap)
            allowed = np.ones((q1 - q0, kvl), bool)
            if batch.causal:
                allowed &= np.tril(np.ones((q1 - q0, kvl), bool), kvl - (q1 - q0))
            if batch.window_left > 0:
                allowed &= np.triu(np.ones((q1 - q0, kvl), bool), kvl - (q1 - q0) - batch.window_left)
            S = np.where(allowed, S, -np.inf)
            for i in range(q1 - q0):
                if kvl == 0 or not np.isfinite(S[i]).any():
                    continue
                L[q0 + i, h] = logsumexp(S[i])
                O[q0 + i, h] = softmax(S[i]) @ V[:, h]
    return O, L


def run_batch(orc, batch):
    return orc.attention(batch.q.float().numpy(), batch.k_pages.float().numpy(),
                         batch.v_pages.float().numpy(), batch.qo_indptr, batch.kv_indptr,
                         batch.kv_indices, batch.last_page_len, batch.num_qo_heads,
                         batch.num_kv_heads, batch.page_size, batch.causal, batch.sm_scale,
                         window_left=batch.window_left, soft_cap=batch.soft_cap)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------


def pin_merge_worked_example(orc):
    """Engineering walkthrough §III.2-3: chunk states and their merge."""
    g = golden("merge_worked_example.json")
    keys, vals, q = g["keys"], [[v, 0.0] for v in g["values"]], g["q"]
    oa, la = run(orc, one_request(keys[:2], vals[:2], q))
    ob, lb = run(orc, one_request(keys[2:], vals[2:], q))
    p, tol = g["printed"], g["printed_precision"]
    assert abs(oa[0] - p["O_A"]) <= tol["O"] and abs(la - p["LSE_A"]) <= tol["LSE"], (oa, la)
    assert abs(ob[0] - p["O_B"]) <= tol["O"] and abs(lb - p["LSE_B"]) <= tol["LSE"], (ob, lb)
    om, lm = orc.merge_states(oa[None], np.array([la]), ob[None], np.array([lb]))
    assert abs(om[0, 0] - p["O_merged"]) <= tol["O"], om
    assert abs(om[0, 0] - p["naive_average_wrong"]) > 1.0
    # the merge equals one-shot attention over all four keys
    oall, lall = run(orc, one_request(keys, vals, q))
    assert abs(om[0, 0] - oall[0]) < 1e-12 and abs(lm[0] - lall) < 1e-12
    # and both equal the closed form sum e^s v / sum e^s, log sum e^s
    s = np.array([1.0, 2.0, 3.0, 4.0])
    assert abs(oall[0] - (np.exp(s) @ np.array(g["values"])) / np.exp(s).sum()) < 1e-12
    assert abs(lall - math.log(np.exp(s).sum())) < 1e-12


def pin_merge_masses(orc):
    """Technical review §3.2: Z_A=2, Z_B=6, O_A=1, O_B=5 merge to 4, LSE log 8."""
    g = golden("merge_masses.json")
    om, lm = orc.merge_states(np.array([[g["O_A"]]]), np.array([math.log(g["Z_A"])]),
                              np.array([[g["O_B"]]]), np.array([math.log(g["Z_B"])]))
    assert abs(om[0, 0] - g["printed"]["O_merged"]) < 1e-12, om
    assert abs(lm[0] - math.log(g["Z_A"] + g["Z_B"])) < 1e-12, lm


def pin_online_two_tiles(orc):
    """Hardware-aware attention notes: scores [0,1,2] in tiles [0,1] and [2]."""
    g = golden("online_softmax_two_tiles.json")
    keys = [[s] for s in g["scores"]]
    vals = [[v] for v in g["values"]]
    (a0, a1), (b0, b1) = g["tiles"]
    oa, la = run(orc, one_request(keys[a0:a1], vals[a0:a1], [1.0]))
    ob, lb = run(orc, one_request(keys[b0:b1], vals[b0:b1], [1.0]))
    # after the first tile: max 1 and sum exp(-1) + 1, i.e. LSE = 1 + log(e^-1 + 1)
    assert abs(la - (g["printed"]["tile1_max"] + math.log(math.exp(-1) + 1))) < 1e-12
    om, lm = orc.merge_states(oa[None], np.array([la]), ob[None], np.array([lb]))
    e = math.e
    closed = (1 + 3 * e + 5 * e * e) / (1 + e + e * e)
    assert abs(om[0, 0] - closed) < 1e-12, (om, closed)
    assert abs(lm[0] - math.log(1 + e + e * e)) < 1e-12


def pin_one_key(orc):
    """One visible key: O = v exactly and LSE = its scaled score."""
    rng = np.random.default_rng(11)
    k, v, q = rng.standard_normal((1, 8)), rng.standard_normal((1, 8)), rng.standard_normal(8)
    o, l = run(orc, one_request(k, v, q, sm_scale=0.37))
    k32, v32, q32 = (np.asarray(x, np.float32).astype(np.float64) for x in (k, v, q))
    assert np.allclose(o, v32[0], rtol=0, atol=1e-15)
    assert abs(l - 0.37 * float(q32 @ k32[0])) < 1e-12


def pin_page_mapping(orc):
    """Technical review §4.1 eq 7: indices [7,2], page 4, token 5 -> row 9."""
    g = golden("page_mapping.json")
    got = orc.physical_row([0, len(g["indices"])], g["indices"], g["page_size"], 0, g["logical_token"])
    assert got == g["physical_token"], got


def pin_toy_bsr(orc):
    """Engineering walkthrough §V.1: tile 0 reads P3,P5,P1; tile 1 reads P2,P4 (B_c = 1)."""
    g = golden("toy_bsr.json")
    for tile, pages in enumerate(g["tile_pages"]):
        rows = [orc.physical_row(g["row_ptr"], g["col_indices"], 1, tile, t) for t in range(len(pages))]
        assert rows == pages, rows


def pin_toy_bsr_attention(orc):
    """Engineering walkthrough §V.1 with B_r = 4: the two query tiles (rows 0-3
    and 4-7) share their tile's page list; each row's attention over the paged
    pool must equal library softmax attention over exactly those pages."""
    g = golden("toy_bsr.json")
    D, br = 4, 4
    rng = np.random.default_rng(13)
    k = rng.standard_normal((6, 1, 1, D)).astype(np.float32)   # pages P0..P5, B_c = 1
    v = rng.standard_normal((6, 1, 1, D)).astype(np.float32)
    q = rng.standard_normal((2 * br, 1, D)).astype(np.float32)
    qo_indptr = [0, br, 2 * br]
    o, lse = orc.attention(q, k, v, qo_indptr, g["row_ptr"], g["col_indices"], [1, 1], 1, 1, 1, False, 0.5)
    for tile, pages in enumerate(g["tile_pages"]):
        rk = np.stack([k[pg, 0, 0] for pg in pages]).astype(np.float64)
        rv = np.stack([v[pg, 0, 0] for pg in pages]).astype(np.float64)
        for r in range(tile * br, (tile + 1) * br):
            s = 0.5 * rk @ q[r, 0].astype(np.float64)
            assert abs(lse[r, 0] - logsumexp(s)) < 1e-12
            assert np.allclose(o[r, 0], softmax(s) @ rv, rtol=0, atol=1e-12)


def pin_bsr_page_table(orc):
    """Overview ⑤: A -> pages 5,1,6; B -> 2; C -> 7,3 (indptr [0,3,4,6]).

    Each request's attention over the paged pool must equal library softmax
    attention over the rows copied out of its pages in the printed order (page
    size 2, last pages partly valid)."""
    g = golden("bsr_page_table.json")
    ps, D = 2, 4
    rng = np.random.default_rng(12)
    k = rng.standard_normal((g["num_pages"], ps, 1, D)).astype(np.float32)
    v = rng.standard_normal((g["num_pages"], ps, 1, D)).astype(np.float32)
    q = rng.standard_normal((3, 1, D)).astype(np.float32)
    last = [1, 2, 1]
    for b, name in enumerate(["A", "B", "C"]):
        pages = g["requests"][name]
        assert pages == g["indices"][g["indptr"][b]:g["indptr"][b + 1]]
        assert orc.physical_row(g["indptr"], g["indices"], ps, b, 0) == pages[0] * ps
    o, lse = orc.attention(q, k, v, np.arange(4), g["indptr"], g["indices"], last, 1, 1, ps, False, 0.5)
    for b, name in enumerate(["A", "B", "C"]):
        pages = g["requests"][name]
        rows_k = np.concatenate([k[p, :, 0] for p in pages])[: (len(pages) - 1) * ps + last[b]]
        rows_v = np.concatenate([v[p, :, 0] for p in pages])[: (len(pages) - 1) * ps + last[b]]
        s = 0.5 * rows_k.astype(np.float64) @ q[b, 0].astype(np.float64)
        assert abs(lse[b, 0] - logsumexp(s)) < 1e-12
        assert np.allclose(o[b, 0], softmax(s) @ rows_v.astype(np.float64), rtol=0, atol=1e-12)


def pin_dense_library(orc):
    """Contiguous batches (GQA, causal bottom-right, ragged, qo < kv) vs library softmax."""
    cases = [
        dict(qo=[1, 1, 1], kv=[5, 1, 9], hq=4, hk=2, ps=4, causal=False),
        dict(qo=[3, 7, 1], kv=[3, 9, 4], hq=6, hk=3, ps=3, causal=True),
        dict(qo=[5, 2], kv=[5, 6], hq=8, hk=2, ps=16, causal=True),
        dict(qo=[4, 1, 6], kv=[4, 7, 6], hq=2, hk=2, ps=1, causal=True),
        dict(qo=[2, 3], kv=[7, 0], hq=4, hk=1, ps=4, causal=False),
    ]
    for i, c in enumerate(cases):
        batch = workloads.paged_batch(100 + i, c["qo"], c["kv"], c["hq"], c["hk"], 8, c["ps"], "f32",
                                      causal=c["causal"], sm_scale=0.3, contiguous=True)
        O, L = run_batch(orc, batch)
        Oe, Le = dense_reference(batch)
        assert np.array_equal(np.isinf(L), np.isinf(Le)), (i, L, Le)
        fin = np.isfinite(Le)
        assert np.allclose(L[fin], Le[fin], rtol=0, atol=1e-12), i
        assert np.allclose(O, Oe, rtol=0, atol=1e-12), i


def pin_soft_cap_one_key(orc):
    """Technical review eq 8 with one key: the state is that key's, O = v and
    LSE = c * tanh(s / c), s the scaled score (closed form)."""
    rng = np.random.default_rng(31)
    D = 8
    q = rng.standard_normal((1, 1, D)).astype(np.float32) * 3
    k = rng.standard_normal((1, 1, 1, D)).astype(np.float32) * 3
    v = rng.standard_normal((1, 1, 1, D)).astype(np.float32)
    for c in (0.5, 2.0, 30.0):
        o, lse = orc.attention(q, k, v, [0, 1], [0, 1], [0], [1], 1, 1, 1, False, 0.7, soft_cap=c)
        s = 0.7 * float(np.dot(q[0, 0].astype(np.float64), k[0, 0, 0].astype(np.float64)))
        assert abs(lse[0, 0] - c * np.tanh(s / c)) < 1e-12
        assert np.allclose(o[0, 0], v[0, 0, 0], rtol=0, atol=1e-15)


def pin_sink_one_key(orc):
    """Attention sink (overview ⑧, the AttentionSink variant: the sink joins the
    softmax's (m, d) as one more logit, the output is normalised by that d) with
    one key and two query heads on one kv head, each with its own sink: closed
    form O_h = v e^{s_h} / (e^{s_h} + e^{sink_h}), LSE_h = log(e^{s_h} + e^{sink_h})."""
    rng = np.random.default_rng(37)
    D = 8
    q = rng.standard_normal((1, 2, D)).astype(np.float32)
    k = rng.standard_normal((1, 1, 1, D)).astype(np.float32)
    v = rng.standard_normal((1, 1, 1, D)).astype(np.float32)
    sink = np.array([0.3, -1.7])
    o, lse = orc.attention(q, k, v, [0, 1], [0, 1], [0], [1], 2, 1, 1, False, 0.6, sink=sink)
    for h in range(2):
        s = 0.6 * float(np.dot(q[0, h].astype(np.float64), k[0, 0, 0].astype(np.float64)))
        assert abs(lse[0, h] - math.log(math.exp(s) + math.exp(sink[h]))) < 1e-12
        w = math.exp(s) / (math.exp(s) + math.exp(sink[h]))
        assert np.allclose(o[0, h], w * v[0, 0, 0].astype(np.float64), rtol=0, atol=1e-14)


def pin_sink_virtual_key(orc):
    """A sink equals one extra key with a zero value row whose score is the sink
    (the sink is a logit without a value): every query gets q[0] = 1 and the extra
    key, placed first, k = (sink / sm_scale, 0, ...), so its score is exactly the
    sink; placing it first keeps the other keys' bottom-right causal visibility."""
    rng = np.random.default_rng(41)
    D, H, sm = 8, 3, 0.5
    sink = np.array([1.5, -0.75, 3.0])
    for causal in (False, True):
        qo, kv = [1, 4, 3], [5, 4, 7]
        n_tok = sum(qo)
        q = rng.standard_normal((n_tok, H, D)).astype(np.float32)
        q[:, :, 0] = 1.0
        ks = [rng.standard_normal((n, H, D)).astype(np.float32) for n in kv]
        vs = [rng.standard_normal((n, H, D)).astype(np.float32) for n in kv]
        virt_k = np.zeros((1, H, D), np.float32)
        virt_k[0, :, 0] = sink / sm
        virt_v = np.zeros((1, H, D), np.float32)

        def batch(extra):
            kp = np.concatenate([np.concatenate(([virt_k] if extra else []) + [k]) for k in ks])
            vp = np.concatenate([np.concatenate(([virt_v] if extra else []) + [v]) for v in vs])
            lens = [n + int(extra) for n in kv]
            return (q, kp.reshape(-1, 1, H, D), vp.reshape(-1, 1, H, D), np.cumsum([0] + qo),
                    np.cumsum([0] + lens), np.arange(sum(lens)), np.ones(len(kv), np.int32), H, H, 1, causal, sm)
        O1, L1 = orc.attention(*batch(False), sink=sink)
        O2, L2 = orc.attention(*batch(True))
        assert np.allclose(L1, L2, rtol=0, atol=1e-12) and np.allclose(O1, O2, rtol=0, atol=1e-12), causal


def pin_sink_limits(orc):
    """A sink of -inf is no sink (bit-identical); a row with no visible key keeps
    O = 0 and gets LSE = sink (the normaliser holds only the sink)."""
    batch = workloads.paged_batch(43, [1, 2, 1], [6, 0, 3], 4, 2, 8, 2, "f32", causal=False)
    args = (batch.q.float().numpy(), batch.k_pages.float().numpy(), batch.v_pages.float().numpy(),
            batch.qo_indptr, batch.kv_indptr, batch.kv_indices, batch.last_page_len, 4, 2, 2, False, 0.35)
    O0, L0 = orc.attention(*args)
    On, Ln = orc.attention(*args, sink=np.full(4, -np.inf))
    assert np.array_equal(O0, On) and np.array_equal(L0, Ln)
    sink = np.array([0.5, -2.0, 1.25, 7.0])
    Os, Ls = orc.attention(*args, sink=sink)
    assert np.all(Os[1:3] == 0) and np.array_equal(Ls[1:3], np.tile(sink, (2, 1)))


def pin_variants_library(orc):
    """Sliding window and soft-cap on contiguous batches vs library routines on
    the explicitly masked, explicitly capped dense scores."""
    cases = [
        dict(qo=[6, 9], kv=[6, 13], hq=4, hk=2, ps=4, causal=True, w=3, cap=0.0),
        dict(qo=[1, 1, 1], kv=[9, 2, 17], hq=4, hk=4, ps=2, causal=True, w=5, cap=0.0),
        dict(qo=[5, 3], kv=[11, 8], hq=6, hk=3, ps=3, causal=False, w=0, cap=1.5),
        dict(qo=[7], kv=[12], hq=2, hk=1, ps=4, causal=True, w=4, cap=2.0),
        dict(qo=[4], kv=[4], hq=2, hk=2, ps=1, causal=False, w=2, cap=0.0),
    ]
    for i, c in enumerate(cases):
        batch = workloads.paged_batch(130 + i, c["qo"], c["kv"], c["hq"], c["hk"], 8, c["ps"], "f32",
                                      causal=c["causal"], sm_scale=0.9, contiguous=True)
        batch.window_left, batch.soft_cap = c["w"], c["cap"]
        O, L = run_batch(orc, batch)
        Oe, Le = dense_reference(batch)
        assert np.array_equal(np.isinf(L), np.isinf(Le)), (i, L, Le)
        fin = np.isfinite(Le)
        assert np.allclose(L[fin], Le[fin], rtol=0, atol=1e-12), i
        assert np.allclose(O, Oe, rtol=0, atol=1e-12), i


def pin_permuted_equals_contiguous(orc):
    """Sparse and dense layouts of the same logical KV give identical fp64
    results (overview ⑥; walkthrough §V.4: the layouts differ only in the loader)."""
    for ps, seed in [(1, 21), (4, 22), (5, 23)]:
        args = (seed, [1, 3, 2], [13, 9, 17], 4, 2, 8, ps, "f32")
        perm = workloads.paged_batch(*args, causal=True, extra_pages=3)
        cont = workloads.paged_batch(*args, causal=True, contiguous=True)
        # same logical values: rebuild the contiguous pool from the permuted one
        k = perm.k_pages.clone()
        v = perm.v_pages.clone()
        cont.q = perm.q
        cont.k_pages = k[np.asarray(perm.kv_indices)]
        cont.v_pages = v[np.asarray(perm.kv_indices)]
        Op, Lp = run_batch(orc, perm)
        Oc, Lc = run_batch(orc, cont)
        assert np.array_equal(Op, Oc) and np.array_equal(Lp, Lc), ps


def pin_causal_prefix(orc):
    """A causal square request: row i equals non-causal attention over keys 0..i."""
    D, ps = 8, 4
    batch = workloads.paged_batch(31, [9], [9], 2, 1, D, ps, "f32", causal=True, sm_scale=0.4)
    O, L = run_batch(orc, batch)
    k = batch.k_pages.float().numpy()
    v = batch.v_pages.float().numpy()
    pages = batch.kv_indices
    for i in range(9):
        n = i + 1
        npg = -(-n // ps)
        Oi, Li = orc.attention(batch.q.float().numpy()[i:i + 1], k, v, [0, 1], [0, npg], pages[:npg],
                               [n - (npg - 1) * ps], 2, 1, ps, False, 0.4)
        assert np.allclose(O[i], Oi[0], rtol=0, atol=1e-12) and np.allclose(L[i], Li[0], rtol=0, atol=1e-12), i


def pin_empty(orc):
    """No visible key: O = 0 and LSE = -inf (the technical review's empty state)."""
    batch = workloads.paged_batch(41, [1, 3], [0, 1], 2, 1, 4, 2, "f32", causal=True)
    O, L = run_batch(orc, batch)
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))
    # causal, qo 3 > kv 1: rows 0 and 1 of request 1 see nothing, row 2 sees key 0
    assert np.all(O[1:3] == 0) and np.all(np.isneginf(L[1:3]))
    assert np.all(np.isfinite(L[3]))


def pin_merge_algebra(orc):
    """Commutative, associative, exact split of a key set, and the empty rule
    (technical review §3.3 Algorithm 1)."""
    rng = np.random.default_rng(51)
    n, D = 64, 16
    O = [rng.standard_normal((n, D)) for _ in range(3)]
    L = [rng.standard_normal(n) * 5 for _ in range(3)]
    ab = orc.merge_states(O[0], L[0], O[1], L[1])
    ba = orc.merge_states(O[1], L[1], O[0], L[0])
    assert np.allclose(ab[0], ba[0], rtol=0, atol=1e-12) and np.allclose(ab[1], ba[1], rtol=0, atol=1e-12)
    ab_c = orc.merge_states(ab[0], ab[1], O[2], L[2])
    bc = orc.merge_states(O[1], L[1], O[2], L[2])
    a_bc = orc.merge_states(O[0], L[0], bc[0], bc[1])
    assert np.allclose(ab_c[0], a_bc[0], rtol=0, atol=1e-12) and np.allclose(ab_c[1], a_bc[1], rtol=0, atol=1e-12)
    empty_o, empty_l = np.zeros((n, D)), np.full(n, -np.inf)
    x = orc.merge_states(O[0], L[0], empty_o, empty_l)
    y = orc.merge_states(empty_o, empty_l, O[0], L[0])
    assert np.array_equal(x[0], O[0]) and np.array_equal(x[1], L[0])
    assert np.array_equal(y[0], O[0]) and np.array_equal(y[1], L[0])
    z = orc.merge_states(empty_o, empty_l, empty_o, empty_l)
    assert np.all(z[0] == 0) and np.all(np.isneginf(z[1]))
    # a request split into two page ranges merges back to the whole
    batch = workloads.paged_batch(52, [1], [23], 4, 2, 8, 4, "f32", sm_scale=0.5)
    Ow, Lw = run_batch(orc, batch)
    args = (batch.q.float().numpy(), batch.k_pages.float().numpy(), batch.v_pages.float().numpy(), [0, 1])
    pages = batch.kv_indices
    O1, L1 = orc.attention(*args, [0, 3], pages[:3], [4], 4, 2, 4, False, 0.5)
    O2, L2 = orc.attention(*args, [0, 3], pages[3:], batch.last_page_len, 4, 2, 4, False, 0.5)
    Om, Lm = orc.merge_states(O1, L1, O2, L2)
    assert np.allclose(Om, Ow, rtol=0, atol=1e-12) and np.allclose(Lm, Lw, rtol=0, atol=1e-12)


def pin_poison_unread(orc):
    """The oracle never reads unused pages or page tails (they hold NaN)."""
    batch = workloads.tiny_decode_f32()
    O, L = run_batch(orc, batch)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))


ALL_PINS = [pin_merge_worked_example, pin_merge_masses, pin_online_two_tiles, pin_one_key,
            pin_page_mapping, pin_toy_bsr, pin_toy_bsr_attention, pin_bsr_page_table, pin_dense_library,
            pin_permuted_equals_contiguous, pin_causal_prefix, pin_empty, pin_merge_algebra,
            pin_poison_unread, pin_soft_cap_one_key, pin_variants_library, pin_sink_one_key,
            pin_sink_virtual_key, pin_sink_limits]
