"""Oracle planner: the load-balanced plan written out in plain Python.

TEST INFRASTRUCTURE ONLY. The product library has its own planner in C++; the
two share no code. Only tests, the package's smoke check and the bench's
CPU-baseline leg import this module.

What it restates, in the order the pages give it (FlashInfer 原理 overview, ⑨
and its worked example; FlashInfer: Making Attention Fit the Serving Workload,
§6.1 eq 10-11 and §6.2 Algorithm 2; Engineering a Customizable, Block-Sparse
Attention Engine, §VIII.2 and §VIII.5):

1. Query tiles. Request b has qo_len_b query positions; with head-group fusion
   each position carries g = H_qo / H_kv rows, so the packed length is
   qo_len_b * g (overview, ⑦; review eq 3). Tiles of T_q packed rows
   (T_q a multiple of g) cover whole positions. Every (tile, kv head) pair is
   one output tile.
2. W = sum over output tiles of kv_len_b (eq 10 with the kv-head factor; the
   kv head is an axis of the work items).
3. L = max(1, ceil(W / C)) (Algorithm 2 step 4 and the overview's worked
   example use the ceiling), then rounded up to a multiple of the page size so
   that no chunk splits a page. An optional s = chunks_per_cta > 1 (not on
   the pages; this build's extension) takes L = ceil(W / (s C)) instead, about
   s chunks per CTA, so that LPT can even out batches of few, equal tiles.
4. Each output tile's visible KV range [lo, v) is cut into chunks of at most
   L tokens from lo on (Algorithm 2 step 5). Non-causal: v = kv_len. Causal
   with bottom-right alignment: v = min(kv_len, last_pos + kv_len - qo_len + 1)
   clamped at 0, last_pos being the tile's largest query position. lo = 0,
   or with a sliding window of window_left > 0 (overview, ⑧: key j visible
   from query i iff j + qo_len + window_left >= kv_len + i) the window's edge
   for the tile's first position, first_pos + kv_len - qo_len - window_left,
   clamped at 0 and rounded down to a page (this build's reading: chunks start
   on page boundaries; the kernels mask the keys before the edge). A tile
   with nothing visible (v <= lo) still gets one empty chunk (0, 0) so that its
   empty state is written.
5. Chunks are sorted by length, longest first, ties broken by the stable id
   (b, tile, kv_head, chunk_start) ascending (Algorithm 2 step 6).
6. A min-heap of (cost, cta_id) starts at (0, c); each chunk goes to the popped
   CTA, whose cost grows by alpha * l_q + beta * chunk_len (eq 11; the
   overview names the cost 2 * qo_len + kv_len, so alpha = 2, beta = 1 by
   default), l_q being the number of query positions in the tile.
7. Reduction map: an output tile with one chunk is written through to the final
   output; one with several chunks gets consecutive partial slots in ascending
   chunk_start order, numbered over output tiles in (b, tile, kv_head) order,
   and its final state is the left-to-right merge of those slots.

Equal shares (schedule="equal"; not on the pages, this build's extension for
batches of few, equal tiles, where LPT over whole tiles leaves CTAs idle):
steps 1-2 as above; then the output tiles' visible ranges [lo, v) are laid end
to end in (b, tile, kv_head) order (tile i starts at P_i, n_i = v_i - lo_i
tokens, V = sum n_i), and CTA c takes the share [x_c, x_{c+1}) with
x_c = floor(c V / C). A cut that falls strictly inside a tile is moved down to
the page boundary at or before it (key lo_i + x - P_i rounded down to a multiple
of page_size), so that chunks start on pages. A tile's chunks are its non-empty
pieces between consecutive cuts, each on the CTA whose share holds it, in
order; a tile with nothing visible gets one empty chunk on the first CTA whose
share ends after P_i (the last CTA if none). Queues hold their chunks in the
order of the concatenation; the reduction map is step 7's. L is reported as
the longest chunk.
"""
from __future__ import annotations

import bisect
import heapq
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Item:
    """One work item: KV chunk [kv_start, kv_end) of output tile (b, tile, kv_head)."""
    b: int
    tile: int
    kv_head: int
    kv_start: int
    kv_end: int
    slot: int  # partial slot, or -1 when written through to the final output


@dataclass(frozen=True)
class Output:
    """One output tile that needs a merge: its partial slots are slot_begin .. slot_begin + n - 1."""
    b: int
    tile: int
    kv_head: int
    slot_begin: int
    n_slots: int


@dataclass
class Plan:
    tile_rows: int
    chunk_len: int          # L
    total_work: int         # W
    queues: list = field(default_factory=list)    # per CTA: list[Item] in execution order
    outputs: list = field(default_factory=list)   # list[Output] in (b, tile, kv_head) order
    num_partials: int = 0
    cta_cost: list = field(default_factory=list)  # final heap cost of each CTA


def kv_len_from_pages(num_pages: int, last_page_len: int, page_size: int) -> int:
    """Tokens of one request: full pages, then the valid part of the last page."""
    return 0 if num_pages <= 0 else (num_pages - 1) * page_size + last_page_len


def tile_positions(qo_len: int, group: int, tile_rows: int, tile: int) -> tuple[int, int]:
    """Query positions [p0, p1) covered by a tile of tile_rows packed rows."""
    per_tile = tile_rows // group
    p0 = tile * per_tile
    return p0, min(qo_len, p0 + per_tile)


def num_tiles(qo_len: int, group: int, tile_rows: int) -> int:
    packed = qo_len * group
    return -(-packed // tile_rows)


def visible_len(qo_len: int, kv_len: int, last_pos: int, causal: bool) -> int:
    if not causal:
        return kv_len
    return max(0, min(kv_len, last_pos + kv_len - qo_len + 1))


def plan(qo_lens, kv_lens, num_kv_heads: int, group: int, tile_rows: int,
         num_ctas: int, page_size: int, causal: bool, alpha: int = 2, beta: int = 1,
         window_left: int = -1, chunks_per_cta: int = 1, schedule: str = "lpt") -> Plan:
    if tile_rows % group != 0:
        raise ValueError("tile_rows must be a multiple of the group size")
    if num_ctas < 1 or page_size < 1:
        raise ValueError("num_ctas and page_size must be positive")
    B = len(qo_lens)

    # 1-2: output tiles and W
    tiles = []  # (b, tile, kv_head, l_q, lo, visible)
    W = 0
    for b in range(B):
        for t in range(num_tiles(qo_lens[b], group, tile_rows)):
            p0, p1 = tile_positions(qo_lens[b], group, tile_rows, t)
            vis = visible_len(qo_lens[b], kv_lens[b], p1 - 1, causal)
            lo = 0
            if window_left > 0:
                lo = max(0, p0 + kv_lens[b] - qo_lens[b] - window_left) // page_size * page_size
                if lo >= vis:
                    lo = vis = 0
            for h in range(num_kv_heads):
                tiles.append((b, t, h, p1 - p0, lo, vis))
                W += kv_lens[b]

    if schedule == "equal":
        return equal_shares(tiles, W, num_ctas, page_size, alpha, beta, tile_rows)
    if schedule != "lpt":
        raise ValueError("schedule must be 'lpt' or 'equal'")

    # 3: chunk length; s = chunks_per_cta > 1 divides it further (s = 1 is the
    # pages' L = ceil(W / C))
    L = max(1, -(-W // (num_ctas * max(1, chunks_per_cta))))
    L = -(-L // page_size) * page_size

    # 4: chunks per output tile, partial slots and the reduction map
    chunks = []  # (b, tile, kv_head, start, end, l_q, slot)
    outputs = []
    next_slot = 0
    for (b, t, h, lq, lo, vis) in tiles:
        bounds = [(s, min(s + L, vis)) for s in range(lo, vis, L)] or [(0, 0)]
        if len(bounds) == 1:
            s, e = bounds[0]
            chunks.append((b, t, h, s, e, lq, -1))
        else:
            outputs.append(Output(b, t, h, next_slot, len(bounds)))
            for i, (s, e) in enumerate(bounds):
                chunks.append((b, t, h, s, e, lq, next_slot + i))
            next_slot += len(bounds)

    # 5: longest first, ties by stable id
    chunks.sort(key=lambda c: (-(c[4] - c[3]), c[0], c[1], c[2], c[3]))

    # 6: LPT assignment with a min-heap keyed by (cost, cta_id)
    heap = [(0, c) for c in range(num_ctas)]
    heapq.heapify(heap)
    queues = [[] for _ in range(num_ctas)]
    for (b, t, h, s, e, lq, slot) in chunks:
        cost, cta = heapq.heappop(heap)
        queues[cta].append(Item(b, t, h, s, e, slot))
        heapq.heappush(heap, (cost + alpha * lq + beta * (e - s), cta))
    cta_cost = [0] * num_ctas
    for cost, cta in heap:
        cta_cost[cta] = cost

    return Plan(tile_rows=tile_rows, chunk_len=L, total_work=W, queues=queues,
                outputs=outputs, num_partials=next_slot, cta_cost=cta_cost)


def equal_shares(tiles, W: int, num_ctas: int, page_size: int, alpha: int, beta: int, tile_rows: int) -> Plan:
    """The equal-share schedule (module docstring) over the output tiles
    (b, tile, kv_head, l_q, lo, visible) of steps 1-2."""
    starts, V = [], 0
    for (_, _, _, _, lo, vis) in tiles:
        starts.append(V)
        V += vis - lo
    cuts = [c * V // num_ctas for c in range(num_ctas + 1)]
    for c in range(1, num_ctas):
        i = bisect.bisect_right(starts, cuts[c]) - 1  # the last tile starting at or before the cut
        while i >= 0 and tiles[i][5] == tiles[i][4]:  # (an empty tile has no inside)
            i -= 1
        if i >= 0:
            lo, vis = tiles[i][4], tiles[i][5]
            P, n = starts[i], vis - lo
            if P < cuts[c] < P + n:
                key = lo + cuts[c] - P
                cuts[c] = P + (key // page_size * page_size - lo)
    queues = [[] for _ in range(num_ctas)]
    outputs = []
    next_slot = 0
    longest = 1
    for i, (b, t, h, lq, lo, vis) in enumerate(tiles):
        P, n = starts[i], vis - lo
        first = bisect.bisect_right(cuts, P, lo=1) - 1  # first CTA whose share ends after P
        if n == 0:
            owner = min(first, num_ctas - 1)
            queues[owner].append(Item(b, t, h, 0, 0, -1))
            continue
        pieces = []
        for c in range(first, num_ctas):
            a, z = max(P, cuts[c]), min(P + n, cuts[c + 1])
            if cuts[c] >= P + n:
                break
            if a < z:
                pieces.append((c, lo + a - P, lo + z - P))
        if len(pieces) > 1:
            outputs.append(Output(b, t, h, next_slot, len(pieces)))
        for k, (c, s, e) in enumerate(pieces):
            queues[c].append(Item(b, t, h, s, e, next_slot + k if len(pieces) > 1 else -1))
            longest = max(longest, e - s)
        if len(pieces) > 1:
            next_slot += len(pieces)
    lq_of = {(b, t): lq for (b, t, _, lq, _, _) in tiles}
    cta_cost = [sum(alpha * lq_of[(it.b, it.tile)] + beta * (it.kv_end - it.kv_start) for it in q) for q in queues]
    return Plan(tile_rows=tile_rows, chunk_len=longest, total_work=W, queues=queues, outputs=outputs,
                num_partials=next_slot, cta_cost=cta_cost)


def makespan_lower_bound(costs, num_ctas: int) -> float:
    """eq 12 of the technical review: T >= max(sum t / C, max t)."""
    if not costs:
        return 0.0
    return max(sum(costs) / num_ctas, max(costs))


def partial_capacity_elements(num_ctas: int, tile_rows: int, num_qo_heads: int, head_dim: int) -> int:
    """eq 13 of the technical review: E_partial <= 2 C T_q H_q (d + 1) scalar elements."""
    return 2 * num_ctas * tile_rows * num_qo_heads * (head_dim + 1)


def prefix_traffic_ratio(n: int, prefix: int, suffix: float) -> float:
    """eq 15 of the technical review: R = n (P + S) / (P + n S)."""
    return n * (prefix + suffix) / (prefix + n * suffix)
