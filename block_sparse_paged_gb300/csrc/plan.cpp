// Host planner: request lengths -> load-balanced work list + reduction map,
// written to a pinned staging buffer and copied once into the device workspace.
//
// Follows the scheduling algorithm of the pages: FlashInfer 原理 overview, ⑨
// (cost function 2 * qo_len + kv_len, chunking at total work / #CTA, longest
// chunk first onto a min-heap of CTA costs, no atomics, write-through for
// unsplit outputs); FlashInfer: Making Attention Fit the Serving Workload,
// §6.1 eq 10-11 and §6.2 Algorithm 2 (ceil(W / C), tie-break by a stable id,
// reduction map); Engineering a Customizable, Block-Sparse Attention Engine,
// §VIII.2 and §VIII.5 (per-CTA queues and the partial -> final index map).
#include <algorithm>
#include <cstring>
#include <functional>
#include <queue>
#include <vector>

#include <cmath>

#include "bsp_internal.h"

namespace bsp {

bool check_problem(const bsp_problem *p) {
    if (!p) return fail(BSP_ERR_INVALID_ARG, "problem is NULL"), false;
    if (p->mode != BSP_MODE_DECODE && p->mode != BSP_MODE_PREFILL)
        return fail(BSP_ERR_INVALID_ARG, "mode must be BSP_MODE_DECODE or BSP_MODE_PREFILL"), false;
    if (p->num_qo_heads < 1 || p->num_kv_heads < 1 || p->num_qo_heads % p->num_kv_heads != 0)
        return fail(BSP_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads"), false;
    if (p->head_dim < 1 || p->page_size < 1)
        return fail(BSP_ERR_INVALID_ARG, "head_dim and page_size must be positive"), false;
    if (p->causal != 0 && p->causal != 1) return fail(BSP_ERR_INVALID_ARG, "causal must be 0 or 1"), false;
    if (p->dtype != BSP_DTYPE_BF16 && p->dtype != BSP_DTYPE_F32)
        return fail(BSP_ERR_INVALID_ARG, "dtype must be BSP_DTYPE_BF16 or BSP_DTYPE_F32"), false;
    if (!(p->logits_soft_cap >= 0.f) || std::isinf(p->logits_soft_cap))
        return fail(BSP_ERR_INVALID_ARG, "logits_soft_cap must be finite and >= 0"), false;
    const int g = p->num_qo_heads / p->num_kv_heads;
    if (p->mode == BSP_MODE_PREFILL && (kPrefillTileRows / 2) % g != 0)
        return fail(BSP_ERR_UNSUPPORTED, "prefill needs 128 % (num_qo_heads / num_kv_heads) == 0"), false;
    return true;
}

// s of L = ceil(W / (s C)); a zero-initialised capacity plans with s = 1
static int chunks_per_cta(const bsp_capacity *c) { return c->chunks_per_cta > 0 ? c->chunks_per_cta : 1; }

bool compute_layout(const bsp_problem *p, const bsp_capacity *c, Layout *L) {
    if (!check_problem(p)) return false;
    if (!c || c->max_batch < 0 || c->num_ctas < 1 || c->max_qo_tokens < 0)
        return fail(BSP_ERR_INVALID_ARG, "capacity needs max_batch >= 0, num_ctas >= 1, max_qo_tokens >= 0"), false;
    if (c->chunks_per_cta < 0 || c->chunks_per_cta > 64)
        return fail(BSP_ERR_INVALID_ARG, "capacity.chunks_per_cta must be in [0, 64]"), false;
    if (c->schedule != BSP_SCHEDULE_LPT && c->schedule != BSP_SCHEDULE_EQUAL_SHARES)
        return fail(BSP_ERR_INVALID_ARG, "capacity.schedule must be BSP_SCHEDULE_LPT or BSP_SCHEDULE_EQUAL_SHARES"), false;
    if (c->max_gather_pages < 0 || (c->max_gather_pages > 0 && p->mode != BSP_MODE_PREFILL))
        return fail(BSP_ERR_INVALID_ARG, "capacity.max_gather_pages must be >= 0, and 0 in decode mode"), false;
    if ((int64_t)c->max_gather_pages * p->page_size > INT32_MAX)
        return fail(BSP_ERR_CAPACITY, "capacity.max_gather_pages x page_size beyond int32 rows"), false;
    const int64_t sC = (int64_t)chunks_per_cta(c) * c->num_ctas;
    const int g = p->num_qo_heads / p->num_kv_heads;
    Layout l;
    l.group = g;
    l.tile_rows = p->mode == BSP_MODE_DECODE ? g : kPrefillTileRows;
    // Query tiles per kv head: decode tiles are one position each; prefill
    // tiles hold 256 / g positions, so sum_b ceil(qo_b g / 256) <= tokens g / 256 + B.
    const int64_t tiles_per_head = p->mode == BSP_MODE_DECODE
        ? c->max_qo_tokens
        : (c->max_qo_tokens * g + kPrefillTileRows - 1) / kPrefillTileRows + c->max_batch;
    l.cap_tiles = tiles_per_head * p->num_kv_heads;
    // Chunks: each tile has max(1, ceil(v / L)) <= 1 + v / L and sum v / L <= W / L <= s C.
    l.cap_items = l.cap_tiles + sC;
    // Split tiles: v > L gives ceil(v / L) <= 2 v / L slots, summing to <= 2 s C.
    l.cap_partials = 2 * sC;
    l.cap_merges = std::min<int64_t>(l.cap_tiles, sC);
    if (l.cap_items > INT32_MAX / 2) return fail(BSP_ERR_CAPACITY, "capacity too large"), false;

    uint64_t off = 0;
    l.off_header = off;
    off += sizeof(DevHeader);
    l.off_queue_indptr = off;
    off = align_up(off + sizeof(int32_t) * (uint64_t)(c->num_ctas + 1), kAlign);
    l.off_items = off;
    off = align_up(off + sizeof(bsp_work_item) * (uint64_t)l.cap_items, kAlign);
    l.off_merges = off;
    off = align_up(off + sizeof(bsp_merge_entry) * (uint64_t)std::max<int64_t>(l.cap_merges, 1), kAlign);
    l.metadata_end = off;
    l.off_status = off;
    off += kAlign;
    l.off_partial_lse = off;
    off = align_up(off + sizeof(float) * (uint64_t)l.cap_partials * l.tile_rows, kAlign);
    l.off_partial_o = off;
    off = align_up(off + sizeof(float) * (uint64_t)l.cap_partials * l.tile_rows * p->head_dim, kAlign);
    if (c->max_gather_pages > 0) {
        const uint64_t esz = p->dtype == BSP_DTYPE_BF16 ? 2 : 4;
        l.gather_pool_bytes = align_up((uint64_t)c->max_gather_pages * p->page_size * p->num_kv_heads *
                                           p->head_dim * esz, kAlign);
        l.off_gather = off;
        off += 2 * l.gather_pool_bytes;
    }
    l.total = off;
    *L = l;
    return true;
}

namespace {

struct Chunk {
    int32_t b, tile, head, start, end, n_pos, slot, merge;
};

int64_t kv_len_of(const int32_t *kv_indptr, const int32_t *last_page_len, int page_size, int b) {
    const int64_t pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    return pages <= 0 ? 0 : (pages - 1) * page_size + last_page_len[b];
}

}  // namespace
}  // namespace bsp

using namespace bsp;

extern "C" size_t bsp_workspace_size(const bsp_problem *problem, const bsp_capacity *capacity) {
    Layout l;
    if (!compute_layout(problem, capacity, &l)) return 0;
    return (size_t)l.total;
}

extern "C" size_t bsp_host_staging_size(const bsp_problem *problem, const bsp_capacity *capacity) {
    Layout l;
    if (!compute_layout(problem, capacity, &l)) return 0;
    return (size_t)l.metadata_end;
}

extern "C" int bsp_plan(const bsp_problem *problem, const bsp_capacity *capacity, int32_t batch,
                        const int32_t *qo_indptr_h, const int32_t *kv_indptr_h,
                        const int32_t *last_page_len_h, int64_t alpha, int64_t beta,
                        void *host_staging, void *workspace, size_t workspace_bytes,
                        bsp_stream_t stream, bsp_plan_info *out) {
    clear_error();
    if (!out) return fail(BSP_ERR_INVALID_ARG, "out is NULL");
    std::memset(out, 0, sizeof(*out));
    Layout lay;
    if (!compute_layout(problem, capacity, &lay)) return last_code();
    const bsp_problem &P = *problem;
    if (batch < 0) return fail(BSP_ERR_INVALID_ARG, "batch < 0");
    if (batch > capacity->max_batch) return fail(BSP_ERR_CAPACITY, "batch exceeds capacity.max_batch");
    if (!kv_indptr_h || (batch > 0 && !last_page_len_h))
        return fail(BSP_ERR_INVALID_ARG, "kv_indptr / last_page_len are NULL");
    if (P.mode == BSP_MODE_PREFILL && !qo_indptr_h)
        return fail(BSP_ERR_INVALID_ARG, "prefill needs qo_indptr");
    if (!host_staging) return fail(BSP_ERR_INVALID_ARG, "host_staging is NULL");
    if (workspace && workspace_bytes < lay.total)
        return fail(BSP_ERR_CAPACITY, "workspace smaller than bsp_workspace_size()");
    if (alpha < 0 || beta < 0) return fail(BSP_ERR_INVALID_ARG, "alpha and beta must be >= 0");

    // ---- validate metadata -------------------------------------------------
    std::vector<int32_t> qo(batch + 1);
    for (int b = 0; b <= batch; ++b) qo[b] = qo_indptr_h ? qo_indptr_h[b] : b;
    if (qo[0] < 0 || kv_indptr_h[0] < 0) return fail(BSP_ERR_INVALID_ARG, "indptr[0] < 0");
    for (int b = 0; b < batch; ++b) {
        if (qo[b + 1] < qo[b]) return fail(BSP_ERR_INVALID_ARG, "qo_indptr is not non-decreasing");
        if (kv_indptr_h[b + 1] < kv_indptr_h[b]) return fail(BSP_ERR_INVALID_ARG, "kv_indptr is not non-decreasing");
        if (kv_indptr_h[b + 1] > kv_indptr_h[b] &&
            (last_page_len_h[b] < 1 || last_page_len_h[b] > P.page_size))
            return fail(BSP_ERR_INVALID_ARG, "last_page_len out of [1, page_size]");
        if (kv_len_of(kv_indptr_h, last_page_len_h, P.page_size, b) > INT32_MAX)
            return fail(BSP_ERR_INVALID_ARG, "kv length beyond int32");
    }
    if ((int64_t)qo[batch] - qo[0] > capacity->max_qo_tokens)
        return fail(BSP_ERR_CAPACITY, "query positions exceed capacity.max_qo_tokens");

    const int g = lay.group, T = lay.tile_rows, per_tile = T / g, H = P.num_kv_heads;
    const int C = capacity->num_ctas;

    // ---- 1-2: tiles and total work W (eq 10 with the kv-head factor) -------
    int64_t W = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t packed = (int64_t)(qo[b + 1] - qo[b]) * g;
        W += (packed + T - 1) / T * kv_len_of(kv_indptr_h, last_page_len_h, P.page_size, b) * H;
    }

    // ---- 3: chunk length L = ceil(W / (s C)), rounded up to whole pages ----
    const int64_t sC = (int64_t)chunks_per_cta(capacity) * C;
    int64_t Lc = std::max<int64_t>(1, (W + sC - 1) / sC);
    Lc = (Lc + P.page_size - 1) / P.page_size * P.page_size;
    Lc = std::min<int64_t>(Lc, (int64_t)INT32_MAX / 2 / P.page_size * P.page_size);

    // ---- 4: each output tile's visible range [lo, vis) -----------------------
    struct TileRange {
        int32_t b, tile, head, p0, p1;
        int64_t lo, vis;
    };
    std::vector<TileRange> tiles;
    for (int b = 0; b < batch; ++b) {
        const int64_t qo_len = qo[b + 1] - qo[b];
        const int64_t kv_len = kv_len_of(kv_indptr_h, last_page_len_h, P.page_size, b);
        const int64_t ntiles = (qo_len * g + T - 1) / T;
        for (int64_t t = 0; t < ntiles; ++t) {
            const int64_t p0 = t * per_tile, p1 = std::min<int64_t>(qo_len, p0 + per_tile);
            int64_t vis = kv_len;  // keys [lo, vis) are visible to some row of the tile
            if (P.causal) vis = std::max<int64_t>(0, std::min<int64_t>(kv_len, (p1 - 1) + kv_len - qo_len + 1));
            int64_t lo = 0;
            if (P.window_left > 0) {
                // the tile's first position sees the most keys from the left; rounded
                // down to a page so that chunks never start inside a page
                lo = std::max<int64_t>(0, p0 + kv_len - qo_len - P.window_left);
                lo = lo / P.page_size * P.page_size;
                if (lo >= vis) lo = vis = 0;  // nothing visible: one empty chunk
            }
            for (int h = 0; h < H; ++h) tiles.push_back({b, (int32_t)t, h, (int32_t)p0, (int32_t)p1, lo, vis});
        }
    }
    if ((int64_t)tiles.size() > lay.cap_items) return fail(BSP_ERR_CAPACITY, "work items exceed capacity");

    std::vector<Chunk> chunks;
    std::vector<bsp_merge_entry> merges;
    std::vector<std::vector<int32_t>> queue(C);
    int32_t next_slot = 0;
    auto add_merge = [&](const TileRange &tr, int64_t n) {
        bsp_merge_entry m{};
        m.b = tr.b; m.tile = tr.tile; m.kv_head = tr.head;
        m.slot_begin = next_slot; m.n_slots = (int32_t)n;
        m.q_tok0 = (int32_t)(qo[tr.b] + tr.p0); m.n_pos = tr.p1 - tr.p0;
        merges.push_back(m);
    };
    auto add_chunk = [&](const TileRange &tr, int64_t start, int64_t end, int64_t i, int64_t n) {
        Chunk ch;
        ch.b = tr.b; ch.tile = tr.tile; ch.head = tr.head;
        ch.start = (int32_t)start; ch.end = (int32_t)end;
        ch.n_pos = tr.p1 - tr.p0;
        ch.slot = n > 1 ? next_slot + (int32_t)i : -1;
        ch.merge = n > 1 ? (int32_t)merges.size() - 1 : -1;
        chunks.push_back(ch);
        return (int32_t)chunks.size() - 1;
    };
    auto check_bounds = [&]() -> bool {
        if ((int64_t)chunks.size() > lay.cap_items) return fail(BSP_ERR_CAPACITY, "work items exceed capacity"), false;
        if ((int64_t)merges.size() > lay.cap_merges)
            return fail(BSP_ERR_CAPACITY, "reduction map exceeds capacity"), false;
        if (next_slot > lay.cap_partials) return fail(BSP_ERR_CAPACITY, "partial states exceed capacity"), false;
        return true;
    };

    if (capacity->schedule == BSP_SCHEDULE_EQUAL_SHARES) {
        // ---- equal shares (not on the pages): the visible ranges end to end in
        // (b, tile, kv_head) order, CTA c takes [floor(c V / C), floor((c+1) V / C)),
        // a cut inside a tile moved down to a page boundary; each tile's pieces
        // between cuts are its chunks, queued in the order of the concatenation.
        std::vector<int64_t> start(tiles.size());
        int64_t V = 0;
        for (size_t i = 0; i < tiles.size(); ++i) {
            start[i] = V;
            V += tiles[i].vis - tiles[i].lo;
        }
        std::vector<int64_t> cut(C + 1);
        size_t ti = 0;
        for (int c = 0; c <= C; ++c) {
            int64_t x = V * c / C;
            if (c > 0 && c < C) {
                while (ti < tiles.size() && start[ti] + (tiles[ti].vis - tiles[ti].lo) <= x) ++ti;
                if (ti < tiles.size() && start[ti] < x) {  // strictly inside tile ti
                    const int64_t key = tiles[ti].lo + (x - start[ti]);
                    x = start[ti] + (key / P.page_size * P.page_size - tiles[ti].lo);
                }
            }
            cut[c] = x;
        }
        int64_t longest = 1;
        int c = 0;
        for (size_t i = 0; i < tiles.size(); ++i) {
            const TileRange &tr = tiles[i];
            const int64_t P0 = start[i], n = tr.vis - tr.lo;
            if (n == 0) {
                int owner = c;
                while (owner < C - 1 && cut[owner + 1] <= P0) ++owner;
                queue[owner].push_back(add_chunk(tr, 0, 0, 0, 1));
                continue;
            }
            // pieces: the shares [cut[c], cut[c+1]) that overlap [P0, P0 + n)
            while (cut[c + 1] <= P0) ++c;
            int64_t pieces = 0;
            for (int cc = c; cc < C && cut[cc] < P0 + n; ++cc)
                if (std::max(P0, cut[cc]) < std::min(P0 + n, cut[cc + 1])) ++pieces;
            if (pieces > 1) add_merge(tr, pieces);
            int64_t k = 0;
            for (int cc = c; cc < C && cut[cc] < P0 + n; ++cc) {
                const int64_t a = std::max(P0, cut[cc]), z = std::min(P0 + n, cut[cc + 1]);
                if (a >= z) continue;
                queue[cc].push_back(add_chunk(tr, tr.lo + a - P0, tr.lo + z - P0, k++, pieces));
                longest = std::max(longest, z - a);
            }
            if (pieces > 1) next_slot += (int32_t)pieces;
        }
        Lc = longest;
        if (!check_bounds()) return last_code();
    } else {
        // ---- 4 (cont.): chunks of at most L tokens, slots, reduction map -----
        for (const TileRange &tr : tiles) {
            const int64_t n = tr.vis == tr.lo ? 1 : (tr.vis - tr.lo + Lc - 1) / Lc;
            if (n > 1) add_merge(tr, n);
            for (int64_t i = 0; i < n; ++i)
                add_chunk(tr, std::min<int64_t>(tr.lo + i * Lc, tr.vis), std::min<int64_t>(tr.lo + (i + 1) * Lc, tr.vis),
                          i, n);
            if (n > 1) next_slot += (int32_t)n;
        }
        if (!check_bounds()) return last_code();

        // ---- 5: longest first; ties by the stable id (b, tile, kv_head, start) --
        std::vector<int32_t> order(chunks.size());
        for (size_t i = 0; i < order.size(); ++i) order[i] = (int32_t)i;
        std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
            const Chunk &a = chunks[x], &c = chunks[y];
            const int32_t la = a.end - a.start, lc = c.end - c.start;
            if (la != lc) return la > lc;
            if (a.b != c.b) return a.b < c.b;
            if (a.tile != c.tile) return a.tile < c.tile;
            if (a.head != c.head) return a.head < c.head;
            return a.start < c.start;
        });

        // ---- 6: LPT onto a min-heap of (cost, cta) ------------------------------
        using Entry = std::pair<int64_t, int32_t>;
        std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
        for (int32_t c = 0; c < C; ++c) heap.push({0, c});
        for (int32_t idx : order) {
            Entry e = heap.top();
            heap.pop();
            const Chunk &ch = chunks[idx];
            queue[e.second].push_back(idx);
            e.first += alpha * ch.n_pos + beta * (int64_t)(ch.end - ch.start);
            heap.push(e);
        }
    }

    // ---- write the staging image ---------------------------------------------
    uint8_t *st = static_cast<uint8_t *>(host_staging);
    DevHeader hdr{};
    hdr.num_items = (int32_t)chunks.size();
    hdr.num_merges = (int32_t)merges.size();
    hdr.num_partials = next_slot;
    hdr.tile_rows = T;
    hdr.group = g;
    hdr.num_ctas = C;
    hdr.chunk_len = (int32_t)Lc;
    std::memcpy(st + lay.off_header, &hdr, sizeof(hdr));
    int32_t *qptr = reinterpret_cast<int32_t *>(st + lay.off_queue_indptr);
    bsp_work_item *items = reinterpret_cast<bsp_work_item *>(st + lay.off_items);
    int32_t n = 0;
    for (int c = 0; c < C; ++c) {
        qptr[c] = n;
        for (int32_t idx : queue[c]) {
            const Chunk &ch = chunks[idx];
            bsp_work_item it{};
            it.b = ch.b; it.tile = ch.tile; it.kv_head = ch.head;
            it.kv_start = ch.start; it.kv_end = ch.end; it.slot = ch.slot;
            it.pos0 = ch.tile * per_tile;
            it.merge = ch.merge;
            it.q_tok0 = qo[ch.b] + it.pos0;
            it.n_pos = ch.n_pos;
            it.qo_len = qo[ch.b + 1] - qo[ch.b];
            it.kv_len = (int32_t)kv_len_of(kv_indptr_h, last_page_len_h, P.page_size, ch.b);
            it.page_base = kv_indptr_h[ch.b];
            items[n++] = it;
        }
    }
    qptr[C] = n;
    if (!merges.empty())
        std::memcpy(st + lay.off_merges, merges.data(), merges.size() * sizeof(bsp_merge_entry));

    // ---- one H2D copy of the used prefix of the metadata, on the caller's stream
    // (header, queue, the n items and, when there are merges, the unused item
    // slots and the merges: the sections are contiguous in that order)
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t err = cudaSuccess;
    const size_t used = merges.empty() ? lay.off_items + sizeof(bsp_work_item) * (size_t)n
                                       : lay.off_merges + sizeof(bsp_merge_entry) * merges.size();
    if (ws) err = cudaMemcpyAsync(ws, st, used, cudaMemcpyHostToDevice, stream);
    if (err != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("plan copy: ") + cudaGetErrorString(err));

    bsp_plan_info &o = *out;
    o.problem = P;
    o.capacity = *capacity;
    o.batch = batch;
    o.tile_rows = T;
    o.group = g;
    o.chunk_len = (int32_t)Lc;
    o.total_work = W;
    o.alpha = alpha;
    o.beta = beta;
    o.num_items = n;
    o.num_merges = (int32_t)merges.size();
    o.num_partials = next_slot;
    o.cap_items = (int32_t)lay.cap_items;
    o.cap_merges = (int32_t)lay.cap_merges;
    o.cap_partials = (int32_t)lay.cap_partials;
    o.off_header = lay.off_header;
    o.off_queue_indptr = lay.off_queue_indptr;
    o.off_items = lay.off_items;
    o.off_merges = lay.off_merges;
    o.off_status = lay.off_status;
    o.off_partial_lse = lay.off_partial_lse;
    o.off_partial_o = lay.off_partial_o;
    o.metadata_bytes = lay.metadata_end;
    o.workspace_bytes = lay.total;
    o.num_qo_tokens = qo[batch];
    o.num_table_pages = kv_indptr_h[batch];
    o.off_gather = lay.off_gather;
    o.gather_pool_bytes = lay.gather_pool_bytes;
    o.valid = ws ? 1 : 2;  // 2: host-only plan, not runnable
    return BSP_OK;
}
