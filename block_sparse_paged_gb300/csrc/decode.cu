// Split-KV paged decode with the g query heads of a kv head fused into one tile,
// and the plan-driven merge of split outputs.
//
// Decode is HBM-bound (FlashInfer: Making Attention Fit the Serving Workload,
// §2.2 eq 2; Engineering a Customizable, Block-Sparse Attention Engine, §II.3-4):
// every byte of K and V is read once, and the g heads that share a kv head reuse
// each loaded KV tile (head-group fusion, technical review eq 3; overview ⑦).
//
// bf16 kernel (one persistent CTA per SM, running its plan queue(s)):
//   - loaders fill a ring of stages through the page table (sparse gather,
//     dense compute: overview ⑥, walkthrough §IV.2 and §V.4). Pages of 8 or
//     more tokens: warp 4 (K) and warp 5 (V) issue one TMA tensor copy per page
//     box (up to 64 rows of one kv head, 128-byte swizzle), page ids read 32
//     boxes at a time one batch ahead. Smaller pages: 16-byte cp.async copies
//     into the same swizzled layout by warps 4-7 (K: 4 and 5, V: 6 and 7, each
//     one half of a stage's tokens: two warps per operand keep twice the copies
//     in flight, 102 -> 89 us on the page-size-1 decode). 3 stages of 128
//     tokens either way. Stages are large because each carries a fixed
//     handshake cost. mbarriers carry the handshake (full: the stage's bytes /
//     every lane's copies landed; empty: the compute warps are done with it);
//     the ring runs across the CTA's work items, so the next item's first
//     stages load while the current one ends.
//   - compute (warps 0..3): each warp takes two 16-token sub-blocks per stage;
//     S = Q K^T and O += P V on the warp-level tensor-core MMA (m16n8k16, rows
//     = the g fused heads), fp32 online softmax in base 2 with the scale folded
//     into log2(e) (walkthrough §II.2); at the end of each item the warps'
//     states are merged in shared memory.
//   - output: the final (O, LSE) when the item is its output's only chunk, else
//     an fp32 partial state in the workspace slot the plan assigned (overview
//     ⑨). A partial is counted in its reduction-map entry with an atomic after
//     a device-scope fence; the CTA whose partial completes the count folds the
//     entry (slots in order, one common maximum) and resets the count, so no
//     CTA ever waits for another and a run is one launch.
//   - every wait is a bounded spin (SM clock cycles); a wait that gives up sets
//     the workspace status word and an abort flag the other warps see, and the
//     CTA returns.
// e4m3 kernel (the same template, kFp8): K / V pools of e4m3 codes (FlashInfer:
// A Customizable Attention Engine for LLM Serving, App. G.4 Table 8), 8 compute
// warps, 256-token stages; codes go from shared memory straight into f16
// fragments of transposed tiles (S^T = K Q^T, O^T = V^T P^T: tokens on the MMA's
// M side, P^T by movmatrix).
// fp32 kernel: CUDA cores, fp32 throughout, same plan and merge.
// Reduction kernel: the reduction map's slots of each split output, merged in
// ascending order with a common maximum (technical review eq 6); used after the
// prefill kernel and by bsp_run_merge_partials.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <climits>
#include <cstring>

#include <cuda_fp16.h>

#include "bsp_internal.h"
#include "device_common.cuh"
#include "sm100.cuh"

namespace bsp {
namespace {

using namespace dev;

constexpr int kDecThreads = 128;            // fp32 kernel
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMmaRows = 16;                 // fused heads per tile (M of the MMA)

// bf16 kernel: warps 0..3 compute, warps 4 and 5 (TMA) or 4..7 (cp.async) load K and V.
constexpr int kConsumers = 4;
constexpr int kTileK = 64;                   // unit of the stage sizes below; the largest page box (rows)
constexpr int kStages = 5;
constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s at 2 GHz: a fault, not a stall
// reduction-map entries a CTA completes and folds after its queue (more are folded at once)
constexpr int kMaxPendingFolds = 32;

// Four e4m3 values (the bytes of x, lowest first) to two f16x2: lo = bytes 0
// and 1, hi = bytes 2 and 3, the lower byte in the lower half. Exact: every
// e4m3 value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t &lo, uint32_t &hi) {
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// Transpose of an 8 x 8 matrix of 16-bit values held as one register per lane
// (lane l: row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// kTma: K and V arrive by TMA tensor copies, one per page box; otherwise by
// 16-byte cp.async; both into 128-byte swizzled [D / 64][rows][128 B] tiles.
// kFp8 (with kTma, D = 128): the ring holds e4m3 rows (128 bytes, one swizzle
// row); the compute warps read the bytes straight into f16 tensor-core
// fragments (no staging copy).
template <int D, bool kTma, bool kFp8 = false, int kNH = 1>
struct DecodeLayout {
    // bf16: 3 stages of 128 tokens (64 KB), each of the 4 compute warps taking
    // two 16-token sub-blocks per stage. Fewer, larger stages: a stage's fixed
    // handshake cost is spread over more bytes.
    // e4m3 with g <= 8: 256-token stages (64 KB), 3 of them, 8 compute warps (two
    // per scheduler, each hiding the other's latency) taking two sub-blocks
    // each (the head-major scratch needs only 8 rows per warp then); g > 8:
    // 128-token stages, 5 of them.
    static constexpr int kTK = kFp8 ? (kNH == 1 ? 4 * kTileK : 2 * kTileK) : 2 * kTileK;
    static constexpr int kS = (kFp8 && kNH == 2) ? kStages : 3;  // ring stages
    static constexpr int kCons = kFp8 ? 8 : 4;                               // compute warps
    static constexpr int kSubB = kTK / (16 * kCons);                         // 16-token sub-blocks per warp and stage
    static constexpr int kScrRows = kFp8 ? 8 * kNH : kMmaRows;               // scratch rows per warp
    static constexpr int kLoad = kTma ? 2 : 4;                               // loader warps
    static constexpr int kThreads = 32 * (kCons + kLoad);
    static constexpr int kElem = kFp8 ? 1 : 2;               // bytes per K/V element in the ring
    // Both gathers fill the same layout: [D * elem / 128 slabs][kTK rows][128 B],
    // 16-byte chunks XOR-swizzled by row (TMA's 128-byte swizzle; the cp.async
    // gather writes the same addresses), so rows need no padding.
    static constexpr int kSlab = kTK * 128;                  // bytes per 128-byte-wide slab
    static constexpr int kTileBytes = kTK * D * kElem;      // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kS * kStageBytes;
    static constexpr int kScratchOff = kRingBytes;
    static constexpr int kScratchBytes = kCons * kScrRows * D * 4;   // per-warp O rows for the item merge
    static constexpr int kStatBytes = kCons * kScrRows * 2 * 4;      // per-warp (m, l)
    static constexpr int kFacBytes = (kCons + 1) * kScrRows * 4;     // per-(warp, row) weights, per-row LSE
    static constexpr int kBarOff = kScratchOff + kScratchBytes + kStatBytes + kFacBytes;
    static constexpr int kNumBars = 2 * kS + 3;             // full[S], empty[S], merge_in, merge_mid, merge_out
    // after the barriers: abort flag, pending-fold count and list
    static constexpr int kFlagBytes = 8 + 4 * (1 + kMaxPendingFolds);
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + kFlagBytes + (kTma ? 1024 : 0);  // TMA: 1024-byte alignment slack
    static_assert(kSmemBytes <= 227 * 1024, "decode ring exceeds shared memory");
    // byte offset of 16-byte chunk c (of D / 8) of ring row r inside a K or V tile
    __device__ static __forceinline__ uint32_t chunk(int r, int c) {
        return (uint32_t)((c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }
};

struct DecodeParams {
    const uint8_t *ws;
    uint64_t off_queue, off_items, off_plse, off_po, off_status;
    const void *q, *k, *v;
    const int32_t *kv_indices;
    void *o;
    float *lse;
    float scale_log2;
    int H_qo, H_kv, g, page_size, tile_rows;
    int box_rows;  // TMA gather: rows per tensor copy (divides page_size and 64)
    uint64_t off_merges;
    int queues_per_cta, num_queues;  // CTA b runs plan queues [b * qpc, min((b + 1) * qpc, C))
    int window_left;         // > 0: keys j < pos + kv_len - qo_len - window_left are masked
    int soft_cap_on;         // scores: tanh(s * cap_in) * cap_out instead of s * scale_log2
    float cap_in, cap_out;   // sm_scale / c and c * log2(e)
    float v_scale;           // output factor (per-tensor V scale of an e4m3 pool; else 1)
    const float *sink;       // per-qo-head sink logits, or null
};

// Fold of one (row r, columns 4 cq .. 4 cq + 3) unit of a reduction-map entry
// (technical review §3.2 eq 6): its slots' partial states into the final O and
// LSE. The partials were written by other CTAs and are read through L2, so the
// fold is latency-bound: the loads of up to 8 slots (their LSEs and float4
// columns) are issued before any is used, one round trip per 8 slots. Up to 8
// slots this is the fold with one common maximum; longer entries fold 8 slots
// at a time, rescaling to the running maximum. Prm: DecodeParams or
// ReduceParams (workspace offsets, outputs, shapes, sinks).
template <int D, typename OutT, typename Prm>
__device__ __forceinline__ void fold_unit(const Prm &p, const bsp_merge_entry &e, int r, int cq) {
    constexpr int kQ = D / 4;     // column quads per row
    constexpr int kBatch = 8;     // slots whose loads are in flight together
    const float *plse = reinterpret_cast<const float *>(p.ws + p.off_plse);
    const float4 *po = reinterpret_cast<const float4 *>(p.ws + p.off_po);
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < e.n_slots; s0 += kBatch) {
        const int ns = min(kBatch, e.n_slots - s0);
        float l[kBatch];
        float4 o[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const size_t prow = (size_t)(e.slot_begin + s0 + j) * p.tile_rows + r;
            l[j] = j < ns ? __ldcg(plse + prow) : -INFINITY;
            o[j] = j < ns ? __ldcg(po + prow * kQ + cq) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mb = M;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) Mb = fmaxf(Mb, l[j]);
        if (Mb == -INFINITY) continue;  // every slot so far empty
        if (M != Mb) {                   // rescale what was folded to the new maximum
            const float f = M == -INFINITY ? 0.f : exp2f((M - Mb) * kLog2e);
            L *= f;
            acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
            M = Mb;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < ns) {
                const float wgt = exp2f((l[j] - M) * kLog2e);
                L += wgt;
                acc.x = fmaf(wgt, o[j].x, acc.x);
                acc.y = fmaf(wgt, o[j].y, acc.y);
                acc.z = fmaf(wgt, o[j].z, acc.z);
                acc.w = fmaf(wgt, o[j].w, acc.w);
            }
        }
    }
    float inv = M != -INFINITY ? 1.f / L : 0.f;
    float lse_row = M != -INFINITY ? M + logf(L) : -INFINITY;
    if (p.sink) inv *= fold_sink(lse_row, p.sink[e.kv_head * p.g + r % p.g]);
    const size_t orow = (size_t)(e.q_tok0 + r / p.g) * p.H_qo + (size_t)e.kv_head * p.g + (r % p.g);
    OutT *dst = static_cast<OutT *>(p.o) + orow * D + cq * 4;
    dst[0] = from_float<OutT>(acc.x * inv);
    dst[1] = from_float<OutT>(acc.y * inv);
    dst[2] = from_float<OutT>(acc.z * inv);
    dst[3] = from_float<OutT>(acc.w * inv);
    if (cq == 0 && p.lse) p.lse[orow] = lse_row;
}

// Merge of one reduction-map entry by threads t = 0..nthreads-1 of the CTA that
// wrote its last partial state: one (row, 4 columns) unit per thread.
template <int D, typename OutT>
__device__ __forceinline__ void merge_entry(const DecodeParams &p, const bsp_merge_entry &e, int t, int nthreads) {
    constexpr int kQ = D / 4;
    const int rows = e.n_pos * p.g;
    for (int u = t; u < rows * kQ; u += nthreads) fold_unit<D, OutT>(p, e, u / kQ, u % kQ);
}

// Status codes the decode kernel writes to the workspace status word.
constexpr int kStatusProducerWait = 0x101;
constexpr int kStatusConsumerWait = 0x102;
constexpr int kStatusMergeWait = 0x103;
constexpr int kStatusProbeWait = 0x1ff;  // wait_probe_kernel

// Bounded mbarrier wait that also gives up as soon as another warp aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status,
                                              int code) {
    if (sm100::mbar_wait_spin(bar, parity, kWaitLimitCycles, abort_flag)) return true;
    if (!*abort_flag) {
        *abort_flag = 1;
        atomicCAS(status, 0, code);
    }
    return false;
}

// One warp waits, with the kernels' bounded spin, on an mbarrier that nothing
// arrives at: the wait gives up after limit_cycles and records the probe code
// in *status the way every kernel wait does (used to test that path).
__global__ void wait_probe_kernel(long long limit_cycles, int *status) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        sm100::mbar_init(b, 1);
        abort_flag = 0;
        sm100::fence_barrier_init();
    }
    __syncthreads();
    if (!sm100::mbar_wait_spin(b, 0, limit_cycles, &abort_flag) && threadIdx.x == 0)
        atomicCAS(status, 0, kStatusProbeWait);
}

// kNH (e4m3 only): 8-head tiles per kv head, ceil(g / 8)
template <int D, bool kTma, bool kFp8 = false, int kNH = 1>
__global__ void __launch_bounds__(DecodeLayout<D, kTma, kFp8, kNH>::kThreads, 1)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const DecodeParams p) {
    static_assert(!kFp8 || (kTma && D == 128), "e4m3 pools: TMA gather, head_dim 128");
    using LY = DecodeLayout<D, kTma, kFp8, kNH>;
    constexpr int kSR = LY::kScrRows;
    constexpr int kStages = LY::kS;
    constexpr int kConsumers = LY::kCons;
    constexpr int kWsThreads = LY::kThreads;
    constexpr int kTK = LY::kTK;
    static_assert(kConsumers == 4 || kConsumers == 8, "four or eight compute warps");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = kTma ? smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023) : smem_raw;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t *queue = reinterpret_cast<const int32_t *>(p.ws + p.off_queue);
    const bsp_work_item *items = reinterpret_cast<const bsp_work_item *>(p.ws + p.off_items);
    int *status = reinterpret_cast<int *>(const_cast<uint8_t *>(p.ws) + p.off_status);
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the merge kernel may get resident now
    const int qb = blockIdx.x * p.queues_per_cta;
    const int it0 = queue[qb], it1 = queue[min(qb + p.queues_per_cta, p.num_queues)];
    if (it0 >= it1) return;  // uniform across the CTA, before any barrier

    const uint32_t sbase = smem_u32(smem);  // 1024-byte aligned in the TMA layout
    const uint32_t full0 = sbase + LY::kBarOff, empty0 = full0 + kStages * 8;
    const uint32_t merge_in = empty0 + kStages * 8, merge_mid = merge_in + 8, merge_out = merge_mid + 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + LY::kBarOff + LY::kNumBars * 8);
    // entries whose count this CTA completed: [0] how many, then their indices
    volatile int *pending = abort_flag + 2;

    // Rows past a chunk's end are never copied: zero the ring once so that
    // they hold finite values (their probabilities are exactly 0).
    for (int i = tid; i < LY::kRingBytes / 16; i += kWsThreads) reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    sm100::fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            sm100::mbar_init(full0 + 8 * s, kTma ? 2 : 32 * LY::kLoad);  // TMA: one per producer warp; else per lane
            sm100::mbar_init(empty0 + 8 * s, kConsumers);
        }
        sm100::mbar_init(merge_in, kConsumers);
        sm100::mbar_init(merge_mid, kConsumers);
        sm100::mbar_init(merge_out, kConsumers);
        *abort_flag = 0;
        pending[0] = 0;
        sm100::fence_barrier_init();
    }
    if (kTma && warp == kConsumers && lane == 0) {
        sm100::prefetch_tmap(&tk);
        sm100::prefetch_tmap(&tv);
    }
    __syncthreads();

    if (kTma && warp >= kConsumers) {
        // ---------------- producers (TMA): warp 4 copies K, warp 5 V --------
        // Lane i issues box i of the stage (box_rows rows of one page, D / 64
        // tensor copies); lane 0 first posts the stage's byte count.
        const bool is_v = warp == kConsumers + 1;
        const CUtensorMap *map = is_v ? &tv : &tk;
        const uint32_t part = is_v ? LY::kTileBytes : 0;
        const int br = p.box_rows;
        const int bps = kTK / br;     // boxes per stage (br is a power of two, 8..64): at most 16
        const int spb = 32 / bps;     // stages whose page ids one warp-wide load covers
        int k = 0;
        for (int it = it0; it < it1 && !*abort_flag; ++it) {
            const bsp_work_item w = items[it];
            const int len = w.kv_end - w.kv_start;
            const int nt = (len + kTK - 1) / kTK;
            // Page ids come in batches of 32 (lane l: box l % bps of stage l / bps of
            // the batch), one batch ahead, so that their latency under a full
            // memory system overlaps the copies instead of gating every stage.
            auto fetch_batch = [&](int b) -> int {
                const int r = (b * spb + lane / bps) * kTK + (lane % bps) * br;
                return r < len ? __ldg(p.kv_indices + w.page_base + (w.kv_start + r) / p.page_size) : 0;
            };
            int cur = nt > 0 ? fetch_batch(0) : 0;
            int nxt = spb < nt ? fetch_batch(1) : 0;
            for (int t = 0; t < nt; ++t, ++k) {
                if (t > 0 && t % spb == 0) {
                    cur = nxt;
                    if (t + spb < nt) nxt = fetch_batch(t / spb + 1);
                }
                const int pg = __shfl_sync(0xffffffffu, cur, (t % spb) * bps + (lane < bps ? lane : 0));
                const int n = min(kTK, len - t * kTK);
                const int nbox = (n + br - 1) / br;
                const int row0 = pg * p.page_size + (w.kv_start + t * kTK + lane * br) % p.page_size;
                const int s = k % kStages;
                const bool ok = wait_or_abort(empty0 + 8 * s, ((k / kStages) & 1) ^ 1, abort_flag, status,
                                              kStatusProducerWait);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) sm100::mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)(nbox * br * D * LY::kElem));
                __syncwarp();
                if (lane < nbox) {
                    const uint32_t dst = sbase + s * LY::kStageBytes + part + (uint32_t)(lane * br * 128);
#pragma unroll
                    for (int h = 0; h < D * LY::kElem / 128; ++h)  // one copy per 128-byte-wide slab
                        sm100::tma_load_3d(dst + h * LY::kSlab, map, full0 + 8 * s, h * (128 / LY::kElem), w.kv_head,
                                           row0);
                }
            }
        }
        return;
    }
    if (!kTma && warp >= kConsumers) {
        // ---------------- producers: warps 4, 5 copy K rows, warps 6, 7 V rows ----
        // Warp 4 (6) takes the first half of each stage's tokens, warp 5 (7) the
        // second. Each lane first turns the page ids of its tokens `lane` and
        // `lane + 32` of the half into byte offsets of their rows (one division
        // each), then every warp instruction copies T = 32 / C whole rows, C =
        // D / 8 chunks of 16 bytes per row, taking the row offsets by shuffle.
        constexpr int C = D / 8, T = 32 / C;
        constexpr int kHalfTK = kTK / 2;  // tokens of a stage per loader warp
        const bool is_v = warp >= kConsumers + 2;
        const int tok_base = ((warp - kConsumers) & 1) * kHalfTK;
        const char *src = static_cast<const char *>(is_v ? p.v : p.k);
        const uint32_t part = is_v ? LY::kTileBytes : 0;
        const int my_chunk = lane % C, my_sub = lane / C;
        int k = 0;
        for (int it = it0; it < it1 && !*abort_flag; ++it) {
            const bsp_work_item w = items[it];
            const int len = w.kv_end - w.kv_start;
            const int nt = (len + kTK - 1) / kTK;
            constexpr int kJ = kHalfTK / 32;  // tokens per lane in this warp's half of a stage
            int pg[kJ];
#pragma unroll
            for (int jj = 0; jj < kJ; ++jj) pg[jj] = 0;
            auto fetch = [&](int t, int (&dst)[kJ]) {
#pragma unroll
                for (int jj = 0; jj < kJ; ++jj) {
                    const int j = tok_base + lane + 32 * jj;
                    const int tok = w.kv_start + t * kTK + j;
                    if (t * kTK + j < len) dst[jj] = __ldg(p.kv_indices + w.page_base + tok / p.page_size);
                }
            };
            if (nt > 0) fetch(0, pg);
            for (int t = 0; t < nt; ++t, ++k) {
                // byte offsets of this lane's two rows, then the next tile's page ids
                uint64_t off[kJ];
#pragma unroll
                for (int jj = 0; jj < kJ; ++jj) {
                    const int tok = w.kv_start + t * kTK + tok_base + lane + 32 * jj;
                    off[jj] = (((uint64_t)pg[jj] * p.page_size + tok % p.page_size) * p.H_kv + w.kv_head) * (D * 2);
                }
                if (t + 1 < nt) fetch(t + 1, pg);
                const int s = k % kStages;
                const bool ok = wait_or_abort(empty0 + 8 * s, ((k / kStages) & 1) ^ 1, abort_flag, status,
                                              kStatusProducerWait);
                if (!__all_sync(0xffffffffu, ok)) break;  // warp-uniform: every lane leaves together
                const int n = min(kTK, len - t * kTK);
                const uint32_t dst = sbase + s * LY::kStageBytes + part;
#pragma unroll
                for (int i = 0; i < kHalfTK / T; ++i) {
                    const int jl = i * T + my_sub;                    // token within this warp's half
                    const int j = tok_base + jl;                      // token within the stage
                    const int half = (i * T) >> 5;                    // same for the whole warp: T divides 32
                    const uint64_t o = __shfl_sync(0xffffffffu, off[half], jl & 31);
                    if (j < n) cp_async_16(dst + LY::chunk(j, my_chunk), src + o + my_chunk * 16, 16);
                }
                // arrive on full[s] once this lane's copies have landed
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(full0 + 8 * s) : "memory");
            }
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");  // nothing may still be in flight when the CTA exits
        return;
    }

    // ---------------- consumers: warps 0..3 ----------------------------------
    const int g = p.g;
    const int r0 = lane >> 2, r1 = r0 + 8;
    float *scratch = reinterpret_cast<float *>(smem + LY::kScratchOff);                      // [warp][16][D]
    float *stats = reinterpret_cast<float *>(smem + LY::kScratchOff + LY::kScratchBytes);  // [warp][16][m, l]
    int k = 0, merges = 0;
    bsp_merge_entry *mmap = reinterpret_cast<bsp_merge_entry *>(const_cast<uint8_t *>(p.ws) + p.off_merges);
    bsp_work_item w_next = items[it0];
    for (int it = it0; it < it1; ++it) {
        // the next item is read at the start of this one, and its query rows are
        // prefetched into L1 before this one's epilogue: neither load then sits
        // at the next item's start
        const bsp_work_item w = w_next;
        if (it + 1 < it1) w_next = items[it + 1];
        const int len = w.kv_end - w.kv_start;
        const int nt = (len + kTK - 1) / kTK;

        if constexpr (kFp8) {
            // e4m3 KV, transposed tiles: S^T = K Q^T and O^T = V^T P^T, so that the
            // 16 tokens of a warp fill the M side of each MMA and the g heads the
            // N side (8 per tile). Dimension order inside the tiles is permuted to
            // match how a lane reads e4m3 bytes (16 at a time):
            //   S^T step kk = 4h + j: k pairs (2c, 2c+1), (2c+8, 2c+9) are dims
            //     64h + 16c + 4j + {0, 1} and {2, 3};
            //   O^T tile dt: rows r and r + 8 are dims 16r + 2dt and 16r + 2dt + 1.
            const int c = lane & 3, qn = lane >> 2;
            uint32_t qf[D / 16][kNH][2];  // Q^T fragments, f16 (exact for bf16 values 2^-14 .. 65504; larger saturate)
            {
                const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q) +
                                          ((size_t)w.q_tok0 * p.H_qo + (size_t)w.kv_head * g) * D;
#pragma unroll
                for (int nh = 0; nh < kNH; ++nh) {
                    const int head = 8 * nh + qn;
                    const uint32_t *qr = reinterpret_cast<const uint32_t *>(qb + (size_t)head * D);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int c2 = (64 * (kk >> 2) + 16 * c + 4 * (kk & 3)) >> 1;  // index in bf16 pairs
                        const uint32_t x = head < g ? __ldg(qr + c2) : 0u, y = head < g ? __ldg(qr + c2 + 1) : 0u;
                        qf[kk][nh][0] = pack_f16_sat(bf16_lo(x), bf16_hi(x));
                        qf[kk][nh][1] = pack_f16_sat(bf16_lo(y), bf16_hi(y));
                    }
                }
            }
            // per head (2c, 2c + 1 of each 8-head tile): running max, this lane's share
            // of the sum (its tokens r, r + 8), O^T accumulators
            float mh[kNH][2], lh[kNH][2], oacc[D / 16][kNH][4];
#pragma unroll
            for (int nh = 0; nh < kNH; ++nh) {
                mh[nh][0] = mh[nh][1] = -INFINITY;
                lh[nh][0] = lh[nh][1] = 0.f;
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) oacc[dt][nh][0] = oacc[dt][nh][1] = oacc[dt][nh][2] = oacc[dt][nh][3] = 0.f;
            }

            for (int t = 0; t < nt; ++t, ++k) {
                const int s = k % kStages;
                const bool ok = wait_or_abort(full0 + 8 * s, (k / kStages) & 1, abort_flag, status, kStatusConsumerWait);
                if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll 1
                for (int sbk = 0; sbk < LY::kSubB; ++sbk) {
                const int row0 = (sbk * kConsumers + warp) * 16;        // this sub-block's first stage row
                const bool last_sb = sbk == LY::kSubB - 1;               // the stage goes back after its loads
                const int valid = min(kTK, len - t * kTK) - row0;      // its tokens
                const int lo_rel = p.window_left > 0
                                       ? w.pos0 + w.kv_len - w.qo_len - p.window_left - (w.kv_start + t * kTK + row0)
                                       : INT_MIN;
                if (valid <= 0) {  // so are the later sub-blocks'
                    if (last_sb) {
                        __syncwarp();
                        if (lane == 0) sm100::mbar_arrive(empty0 + 8 * s);
                    }
                    continue;
                }
                const uint32_t kb = sbase + s * LY::kStageBytes, vb = kb + LY::kTileBytes;
                // K rows r, r + 8 (dims 64h + 16c .. + 15); V rows 2c, 2c + 1, 2c + 8,
                // 2c + 9 (dims 16r .. + 15), zero past the chunk end; then the stage is free
                uint4 kw[2][2], vw[4];
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int R = row0 + 8 * t2 + qn;
                        kw[t2][h] = sm100::ld_shared_v4(kb + R * 128 + (((4 * h + c) ^ (R & 7)) << 4));
                    }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = 2 * c + (i & 1) + 8 * (i >> 1), R = row0 + rr;
                    vw[i] = sm100::ld_shared_v4(vb + R * 128 + ((qn ^ (R & 7)) << 4));
                }
                if (valid < 16) {  // the chunk ends inside this warp's rows (warp-uniform)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (2 * c + (i & 1) + 8 * (i >> 1) >= valid) vw[i] = make_uint4(0, 0, 0, 0);
                }
                if (last_sb) {
                    __syncwarp();
                    if (lane == 0) sm100::mbar_arrive(empty0 + 8 * s);
                }

                // S^T: two accumulators per head tile (even / odd kk) to halve the chain
                float st[kNH][2][4];
#pragma unroll
                for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
                    for (int e = 0; e < 2; ++e) st[nh][e][0] = st[nh][e][1] = st[nh][e][2] = st[nh][e][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int h = kk >> 2, j = kk & 3;
                    const uint32_t w0 = j == 0 ? kw[0][h].x : j == 1 ? kw[0][h].y : j == 2 ? kw[0][h].z : kw[0][h].w;
                    const uint32_t w1 = j == 0 ? kw[1][h].x : j == 1 ? kw[1][h].y : j == 2 ? kw[1][h].z : kw[1][h].w;
                    uint32_t a[4];  // rows r, r + 8 x dims {0, 1}, then {2, 3}
                    e4m3x4_to_f16x4(w0, a[0], a[2]);
                    e4m3x4_to_f16x4(w1, a[1], a[3]);
#pragma unroll
                    for (int nh = 0; nh < kNH; ++nh) mma_f16_16816(st[nh][kk & 1], a, qf[kk][nh][0], qf[kk][nh][1]);
                }
                // scale, mask (token r: values 0, 1; token r + 8: values 2, 3), per-head max
                uint32_t pb[kNH][2];
#pragma unroll
                for (int nh = 0; nh < kNH; ++nh) {
                    float sv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float v = st[nh][0][e] + st[nh][1][e];
                        const int tk = qn + 8 * (e >> 1);
                        const float x = p.soft_cap_on ? tanh_ex2(v * p.cap_in) * p.cap_out : v * p.scale_log2;
                        sv[e] = (tk < valid && tk >= lo_rel) ? x : -INFINITY;
                    }
                    float mx0 = fmaxf(sv[0], sv[2]), mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                    const float n0 = fmaxf(mh[nh][0], mx0), n1 = fmaxf(mh[nh][1], mx1);
                    const float ref0 = n0 == -INFINITY ? 0.f : n0, ref1 = n1 == -INFINITY ? 0.f : n1;
                    const float a0 = exp2f(mh[nh][0] - ref0), a1 = exp2f(mh[nh][1] - ref1);
                    mh[nh][0] = n0;
                    mh[nh][1] = n1;
                    const float p0 = exp2f(sv[0] - ref0), p1 = exp2f(sv[1] - ref1);
                    const float p2 = exp2f(sv[2] - ref0), p3 = exp2f(sv[3] - ref1);
                    lh[nh][0] = lh[nh][0] * a0 + (p0 + p2);
                    lh[nh][1] = lh[nh][1] * a1 + (p1 + p3);
                    if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                        for (int dt = 0; dt < D / 16; ++dt) {
                            oacc[dt][nh][0] *= a0; oacc[dt][nh][1] *= a1;
                            oacc[dt][nh][2] *= a0; oacc[dt][nh][3] *= a1;
                        }
                    }
                    // P (tokens x heads) as two 8 x 8 f16 blocks -> transposed: P^T fragments
                    pb[nh][0] = movmatrix_trans(pack_f16_sat(p0, p1));
                    pb[nh][1] = movmatrix_trans(pack_f16_sat(p2, p3));
                }
                // O^T += V^T P^T: word m of the V rows feeds dim tiles 2m and 2m + 1
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t va = m == 0 ? vw[0].x : m == 1 ? vw[0].y : m == 2 ? vw[0].z : vw[0].w;
                    const uint32_t vb2 = m == 0 ? vw[1].x : m == 1 ? vw[1].y : m == 2 ? vw[1].z : vw[1].w;
                    const uint32_t vc = m == 0 ? vw[2].x : m == 1 ? vw[2].y : m == 2 ? vw[2].z : vw[2].w;
                    const uint32_t vd = m == 0 ? vw[3].x : m == 1 ? vw[3].y : m == 2 ? vw[3].z : vw[3].w;
                    const uint32_t lo01 = prmt(va, vb2, 0x5140), lo23 = prmt(va, vb2, 0x7362);
                    const uint32_t hi01 = prmt(vc, vd, 0x5140), hi23 = prmt(vc, vd, 0x7362);
                    uint32_t a_e[4], a_o[4];
                    e4m3x4_to_f16x4(lo01, a_e[0], a_e[1]);
                    e4m3x4_to_f16x4(hi01, a_e[2], a_e[3]);
                    e4m3x4_to_f16x4(lo23, a_o[0], a_o[1]);
                    e4m3x4_to_f16x4(hi23, a_o[2], a_o[3]);
#pragma unroll
                    for (int nh = 0; nh < kNH; ++nh) {
                        mma_f16_16816(oacc[2 * m][nh], a_e, pb[nh][0], pb[nh][1]);
                        mma_f16_16816(oacc[2 * m + 1][nh], a_o, pb[nh][0], pb[nh][1]);
                    }
                }
                }  // sub-blocks
            }

            // ---- this warp's state per head -> stats / scratch rows (heads) ----
#pragma unroll
            for (int nh = 0; nh < kNH; ++nh) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    lh[nh][0] += __shfl_xor_sync(0xffffffffu, lh[nh][0], o);
                    lh[nh][1] += __shfl_xor_sync(0xffffffffu, lh[nh][1], o);
                }
                const int h0 = 8 * nh + 2 * c;
                if (qn == 0) {
                    stats[(warp * kSR + h0) * 2 + 0] = mh[nh][0];
                    stats[(warp * kSR + h0) * 2 + 1] = lh[nh][0];
                    stats[(warp * kSR + h0 + 1) * 2 + 0] = mh[nh][1];
                    stats[(warp * kSR + h0 + 1) * 2 + 1] = lh[nh][1];
                }
                float *s0 = scratch + (warp * kSR + h0) * D + 16 * qn;
                float *s1 = s0 + D;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {
                    *reinterpret_cast<float4 *>(s0 + 4 * i) =
                        make_float4(oacc[2 * i][nh][0], oacc[2 * i][nh][2], oacc[2 * i + 1][nh][0], oacc[2 * i + 1][nh][2]);
                    *reinterpret_cast<float4 *>(s1 + 4 * i) =
                        make_float4(oacc[2 * i][nh][1], oacc[2 * i][nh][3], oacc[2 * i + 1][nh][1], oacc[2 * i + 1][nh][3]);
                }
            }
        } else {
            // Q fragments of the g fused rows (rows >= g are zero)
            uint32_t qa[D / 16][4];
            {
                const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q) +
                                          ((size_t)w.q_tok0 * p.H_qo + (size_t)w.kv_head * g) * D;
                const uint32_t *q0 = reinterpret_cast<const uint32_t *>(qb + (size_t)r0 * D);
                const uint32_t *q1 = reinterpret_cast<const uint32_t *>(qb + (size_t)r1 * D);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c2 = (kk * 16 + 2 * (lane & 3)) >> 1;  // index in bf16 pairs
                    qa[kk][0] = r0 < g ? __ldg(q0 + c2) : 0u;
                    qa[kk][1] = r1 < g ? __ldg(q1 + c2) : 0u;
                    qa[kk][2] = r0 < g ? __ldg(q0 + c2 + 4) : 0u;
                    qa[kk][3] = r1 < g ? __ldg(q1 + c2 + 4) : 0u;
                }
            }
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
            float acc[D / 8][4];
#pragma unroll
            for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

            for (int t = 0; t < nt; ++t, ++k) {
                const int s = k % kStages;
                const bool ok = wait_or_abort(full0 + 8 * s, (k / kStages) & 1, abort_flag, status, kStatusConsumerWait);
                if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll 1
                for (int sbk = 0; sbk < LY::kSubB; ++sbk) {
                const int row0 = (sbk * kConsumers + warp) * 16;        // this sub-block's first stage row
                const int valid = min(kTK, len - t * kTK) - row0;      // its tokens
                // sliding window: tokens of this warp before the window's edge (the chunk
                // starts on a page boundary at or before it) are masked
                const int lo_rel = p.window_left > 0
                                       ? w.pos0 + w.kv_len - w.qo_len - p.window_left - (w.kv_start + t * kTK + row0)
                                       : INT_MIN;
                if (valid > 0) {
                    const uint32_t kb = sbase + s * LY::kStageBytes;
                    const uint32_t vb = kb + LY::kTileBytes;
                    if (kTma && valid < 16) {
                        // whole page boxes were copied: V rows of this warp past the chunk
                        // end may hold anything; zero them so that P = 0 meets finite values
                        for (int e = lane; e < (16 - valid) * (D / 8); e += 32) {
                            const int row = row0 + valid + e / (D / 8);
                            *reinterpret_cast<uint4 *>(smem + (vb - sbase) + LY::chunk(row, e % (D / 8))) =
                                make_uint4(0, 0, 0, 0);
                        }
                        __syncwarp();
                    }
                    float sc[2][4];
#pragma unroll
                    for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                    {
                        const int mi = lane >> 3;
                        const int row = row0 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            uint32_t b0, b1, b2, b3;
                            ldmatrix_x4(kb + LY::chunk(row, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                            mma_bf16_16816(sc[0], qa[kk], b0, b1);
                            mma_bf16_16816(sc[1], qa[kk], b2, b3);
                        }
                    }
                    // scale into base 2, mask tokens past the chunk end
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int tk = n * 8 + 2 * (lane & 3) + (c & 1);
                            const float x = p.soft_cap_on ? tanh_ex2(sc[n][c] * p.cap_in) * p.cap_out : sc[n][c] * p.scale_log2;
                            sc[n][c] = (tk < valid && tk >= lo_rel) ? x : -INFINITY;
                        }
                        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
                        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
                    }
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                    const float ref0 = n0 == -INFINITY ? 0.f : n0, ref1 = n1 == -INFINITY ? 0.f : n1;
                    const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
                    m0 = n0;
                    m1 = n1;
                    float ps[2][4];
                    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        ps[n][0] = exp2f(sc[n][0] - ref0);
                        ps[n][1] = exp2f(sc[n][1] - ref0);
                        ps[n][2] = exp2f(sc[n][2] - ref1);
                        ps[n][3] = exp2f(sc[n][3] - ref1);
                        sum0 += ps[n][0] + ps[n][1];
                        sum1 += ps[n][2] + ps[n][3];
                    }
                    l0 = l0 * a0 + sum0;
                    l1 = l1 * a1 + sum1;
                    if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                        for (int n = 0; n < D / 8; ++n) {
                            acc[n][0] *= a0; acc[n][1] *= a0;
                            acc[n][2] *= a1; acc[n][3] *= a1;
                        }
                    }
                    uint32_t pa[4];
                    pa[0] = pack_bf16(ps[0][0], ps[0][1]);
                    pa[1] = pack_bf16(ps[0][2], ps[0][3]);
                    pa[2] = pack_bf16(ps[1][0], ps[1][1]);
                    pa[3] = pack_bf16(ps[1][2], ps[1][3]);
                    {
                        const int mi = lane >> 3;
                        const int row = row0 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                        for (int nd = 0; nd < D / 16; ++nd) {
                            uint32_t b0, b1, b2, b3;
                            ldmatrix_x4_trans(vb + LY::chunk(row, 2 * nd + (mi >> 1)), b0, b1, b2, b3);
                            mma_bf16_16816(acc[2 * nd], pa, b0, b1);
                            mma_bf16_16816(acc[2 * nd + 1], pa, b2, b3);
                        }
                    }
                }
                }  // sub-blocks
                if (kTma) sm100::fence_proxy_async_smem();  // generic writes above before the next tensor copy
                __syncwarp();
                if (lane == 0) sm100::mbar_arrive(empty0 + 8 * s);
            }

            // ---- merge the four warps' states; write the output or a partial ----
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            if ((lane & 3) == 0) {
                stats[(warp * kSR + r0) * 2 + 0] = m0;
                stats[(warp * kSR + r0) * 2 + 1] = l0;
                stats[(warp * kSR + r1) * 2 + 0] = m1;
                stats[(warp * kSR + r1) * 2 + 1] = l1;
            }
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                const int col = n * 8 + 2 * (lane & 3);
                *reinterpret_cast<float2 *>(scratch + (warp * kSR + r0) * D + col) = make_float2(acc[n][0], acc[n][1]);
                *reinterpret_cast<float2 *>(scratch + (warp * kSR + r1) * D + col) = make_float2(acc[n][2], acc[n][3]);
            }
        }
        if (warp == 0 && it + 1 < it1 && lane * 128 < g * D * 2) {  // the next item's g query rows
            const char *qn = static_cast<const char *>(p.q) +
                             ((size_t)w_next.q_tok0 * p.H_qo + (size_t)w_next.kv_head * g) * D * 2 + lane * 128;
            asm volatile("prefetch.global.L1 [%0];\n" ::"l"(qn));
        }
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(merge_in);
        if (!__all_sync(0xffffffffu, wait_or_abort(merge_in, merges & 1, abort_flag, status, kStatusMergeWait))) return;
        // Combination weights, once per row: warp ww's state of row r enters as
        // fac[ww][r] = 2^(m_ww - M) / L (times the output scale, and the sink's
        // factor for a final row); rlse[r] is the row's LSE.
        float *fac = stats + kConsumers * kSR * 2;  // [warp][row]
        float *rlse = fac + kConsumers * kSR;       // [row]
        const int ct = warp * 32 + lane;
        if (ct < g) {
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kConsumers; ++ww) M = fmaxf(M, stats[(ww * kSR + ct) * 2]);
            float f[kConsumers], L = 0.f;
#pragma unroll
            for (int ww = 0; ww < kConsumers; ++ww) {
                f[ww] = M != -INFINITY ? exp2f(stats[(ww * kSR + ct) * 2] - M) : 0.f;
                L += stats[(ww * kSR + ct) * 2 + 1] * f[ww];
            }
            float inv = M != -INFINITY ? p.v_scale / L : 0.f;
            float lse_v = M != -INFINITY ? (M + log2f(L)) * kLn2 : -INFINITY;
            if (w.slot < 0 && p.sink) inv *= fold_sink(lse_v, p.sink[w.kv_head * g + ct]);
#pragma unroll
            for (int ww = 0; ww < kConsumers; ++ww) fac[ww * kSR + ct] = f[ww] * inv;
            rlse[ct] = lse_v;
        }
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(merge_mid);
        if (!__all_sync(0xffffffffu, wait_or_abort(merge_mid, merges & 1, abort_flag, status, kStatusMergeWait))) return;
        // one (row, 4 columns) unit per thread and pass: the warps' float4s
        // weighted and summed, then 4 bf16 of the output or a float4 of the partial
        for (int u = ct; u < g * (D / 4); u += kConsumers * 32) {
            const int row = u / (D / 4), cq = u - row * (D / 4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ww = 0; ww < kConsumers; ++ww) {
                const float fw = fac[ww * kSR + row];
                const float4 x = reinterpret_cast<const float4 *>(scratch + (ww * kSR + row) * D)[cq];
                acc.x = fmaf(fw, x.x, acc.x);
                acc.y = fmaf(fw, x.y, acc.y);
                acc.z = fmaf(fw, x.z, acc.z);
                acc.w = fmaf(fw, x.w, acc.w);
            }
            if (w.slot < 0) {
                const size_t orow = (size_t)w.q_tok0 * p.H_qo + (size_t)w.kv_head * g + row;
                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.o) + orow * D + cq * 4) =
                    make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
                if (cq == 0 && p.lse) p.lse[orow] = rlse[row];
            } else {
                const size_t prow = (size_t)w.slot * p.tile_rows + row;
                reinterpret_cast<float4 *>(const_cast<uint8_t *>(p.ws) + p.off_po)[prow * (D / 4) + cq] = acc;
                if (cq == 0) reinterpret_cast<float *>(const_cast<uint8_t *>(p.ws) + p.off_plse)[prow] = rlse[row];
            }
        }
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(merge_out);
        if (!__all_sync(0xffffffffu, wait_or_abort(merge_out, merges & 1, abort_flag, status, kStatusMergeWait))) return;
        ++merges;
        if (w.slot >= 0 && warp == 0 && lane == 0) {
            // Split output: count this partial in its reduction-map entry. Every
            // consumer thread wrote its partial rows before merge_out; one gpu-scope
            // fence here orders them all (fences are cumulative) before the count.
            // The CTA whose partial completes the count folds the entry after its
            // queue (nobody waits for another CTA, and no warp waits here for the
            // atomic's round trip).
            __threadfence();
            const int prev = atomicAdd(&mmap[w.merge].arrived, 1);
            if (prev == mmap[w.merge].n_slots - 1) {
                __threadfence();  // acquire: the other CTAs' partials, counted before their arrivals
                const int n = pending[0];
                if (n < kMaxPendingFolds) {
                    pending[1 + n] = w.merge;
                    pending[0] = n + 1;
                } else {  // list full: fold this entry now, by this thread alone
                    merge_entry<D, __nv_bfloat16>(p, mmap[w.merge], 0, 1);
                    mmap[w.merge].arrived = 0;  // ready for the next run of the plan
                }
            }
        }
    }
    // ---- folds of the entries this CTA completed ----------------------------
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(merge_in);
    if (!__all_sync(0xffffffffu, wait_or_abort(merge_in, merges & 1, abort_flag, status, kStatusMergeWait))) return;
    const int n_pending = pending[0];
    for (int i = 0; i < n_pending; ++i) {
        const int ei = pending[1 + i];
        merge_entry<D, __nv_bfloat16>(p, mmap[ei], warp * 32 + lane, kConsumers * 32);
        if (warp == 0 && lane == 0) mmap[ei].arrived = 0;  // ready for the next run of the plan
    }
}

// fp32 decode: CUDA-core fp32 arithmetic, one warp per fused row, lanes over
// head_dim (D / 32 elements each), keys streamed from global memory.
template <int D>
__global__ void __launch_bounds__(kDecThreads) decode_f32_kernel(const DecodeParams p) {
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t *queue = reinterpret_cast<const int32_t *>(p.ws + p.off_queue);
    const bsp_work_item *items = reinterpret_cast<const bsp_work_item *>(p.ws + p.off_items);
    const float *qg = static_cast<const float *>(p.q);
    const float *kg = static_cast<const float *>(p.k);
    const float *vg = static_cast<const float *>(p.v);
    bsp_merge_entry *mmap = reinterpret_cast<bsp_merge_entry *>(const_cast<uint8_t *>(p.ws) + p.off_merges);
    __shared__ int s_last;
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the merge kernel may get resident now
    const int qb = blockIdx.x * p.queues_per_cta;
    for (int it = queue[qb]; it < queue[min(qb + p.queues_per_cta, p.num_queues)]; ++it) {
        const bsp_work_item w = items[it];
        for (int row = warp; row < p.g; row += kDecWarps) {
            const size_t qrow = (size_t)w.q_tok0 * p.H_qo + (size_t)w.kv_head * p.g + row;
            float qr[E], acc[E];
#pragma unroll
            for (int i = 0; i < E; ++i) { qr[i] = qg[qrow * D + lane + 32 * i]; acc[i] = 0.f; }
            float m = -INFINITY, l = 0.f;
            const int t_lo = p.window_left > 0 ? max(w.kv_start, w.pos0 + w.kv_len - w.qo_len - p.window_left)
                                               : w.kv_start;  // sliding window's edge
            for (int t = t_lo; t < w.kv_end; ++t) {
                const int page = __ldg(p.kv_indices + w.page_base + t / p.page_size);
                const size_t kr = ((size_t)page * p.page_size + t % p.page_size) * p.H_kv + w.kv_head;
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < E; ++i) dot = fmaf(qr[i], kg[kr * D + lane + 32 * i], dot);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                const float x = p.soft_cap_on ? tanh_ex2(dot * p.cap_in) * p.cap_out : dot * p.scale_log2;
                const float mn = fmaxf(m, x);
                const float a = exp2f(m - mn), pe = exp2f(x - mn);
                l = l * a + pe;
#pragma unroll
                for (int i = 0; i < E; ++i) acc[i] = fmaf(pe, vg[kr * D + lane + 32 * i], acc[i] * a);
                m = mn;
            }
            const bool empty = !(l > 0.f);  // no visible key (empty chunk, or all before the window)
            float inv = empty ? 0.f : 1.f / l;
            float lse_v = empty ? -INFINITY : (m + log2f(l)) * kLn2;
            if (w.slot < 0) {
                if (p.sink) inv *= fold_sink(lse_v, p.sink[w.kv_head * p.g + row]);
                float *o = static_cast<float *>(p.o) + qrow * D;
#pragma unroll
                for (int i = 0; i < E; ++i) o[lane + 32 * i] = acc[i] * inv;
                if (lane == 0 && p.lse) p.lse[qrow] = lse_v;
            } else {
                const size_t prow = (size_t)w.slot * p.tile_rows + row;
                float *po = reinterpret_cast<float *>(const_cast<uint8_t *>(p.ws) + p.off_po) + prow * D;
#pragma unroll
                for (int i = 0; i < E; ++i) po[lane + 32 * i] = acc[i] * inv;
                if (lane == 0) reinterpret_cast<float *>(const_cast<uint8_t *>(p.ws) + p.off_plse)[prow] = lse_v;
            }
        }
        if (w.slot >= 0) {
            // split output: the CTA whose partial completes the count merges them all
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_last = atomicAdd(&mmap[w.merge].arrived, 1) == mmap[w.merge].n_slots - 1;
            __syncthreads();
            if (s_last) {
                __threadfence();
                const bsp_merge_entry e = mmap[w.merge];
                merge_entry<D, float>(p, e, threadIdx.x, kDecWarps * 32);
                if (threadIdx.x == 0) mmap[w.merge].arrived = 0;  // ready for the next run of the plan
            }
            __syncthreads();
        }
    }
}

// Merge of split outputs: one warp per (reduction-map entry, fused row).
struct ReduceParams {
    const uint8_t *ws;
    uint64_t off_header, off_merges, off_plse, off_po;
    void *o;
    float *lse;
    int H_qo, g, tile_rows;
    const float *sink;  // per-qo-head sink logits, or null
};

template <int D, typename OutT>
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceParams p) {
    // Launched as a programmatic dependent of the attention kernel: it may be
    // resident before that kernel ends, and waits here until its writes
    // (partial states, the header) are complete and visible.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    constexpr int kQ = D / 4;
    const DevHeader *hdr = reinterpret_cast<const DevHeader *>(p.ws + p.off_header);
    const bsp_merge_entry *merges = reinterpret_cast<const bsp_merge_entry *>(p.ws + p.off_merges);
    // one (row, 4 columns) unit per thread and turn; the grid is sized to the
    // plan's units when launched, and strides over any plan's
    const long long units = (long long)hdr->num_merges * p.tile_rows * kQ;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const long long rr = u / kQ;
        const int cq = (int)(u - rr * kQ);
        const bsp_merge_entry &e = merges[rr / p.tile_rows];
        const int r = (int)(rr % p.tile_rows);
        if (r < e.n_pos * p.g) fold_unit<D, OutT>(p, e, r, cq);
    }
}

int num_sms_of_current_device(int *dev_out) {
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (!sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        sms[dev] = n;
    }
    if (dev_out) *dev_out = dev;
    return sms[dev];
}

template <int D, bool kTma, bool kFp8 = false, int kNH = 1>
int launch_decode_bf16(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                       cudaStream_t stream) {
    static bool configured[64] = {false};
    int dev = 0;
    if (num_sms_of_current_device(&dev) < 0) return fail(BSP_ERR_CUDA, "no current CUDA device");
    constexpr int kSmem = DecodeLayout<D, kTma, kFp8, kNH>::kSmemBytes;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<D, kTma, kFp8, kNH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("decode smem attribute: ") + cudaGetErrorString(e));
        configured[dev] = true;
    }
    decode_bf16_kernel<D, kTma, kFp8, kNH><<<grid, DecodeLayout<D, kTma, kFp8, kNH>::kThreads, kSmem, stream>>>(tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("decode launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

template <int D>
int launch_decode_f32(const DecodeParams &p, int grid, cudaStream_t stream) {
    decode_f32_kernel<D><<<grid, kDecThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("decode launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

template <int D, typename OutT>
int launch_reduce_t(const ReduceParams &p, int64_t units, cudaStream_t stream) {
    const int sms = num_sms_of_current_device(nullptr);
    if (sms < 0) return fail(BSP_ERR_CUDA, "no current CUDA device");
    // one unit per thread for this plan (every load in flight at once), at
    // least two CTAs per SM and at most 64
    const int64_t want = (units + 255) / 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<int64_t>(2 * sms, std::min<int64_t>(want, 64 * (int64_t)sms)));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap its launch with the kernel before it
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, reduce_kernel<D, OutT>, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("reduce launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

}  // namespace

int decode_ctas_per_sm(int head_dim, int dtype) {
    if (dtype != BSP_DTYPE_BF16) return 4;
    return 1;  // a ring of 128-token K+V stages and the merge scratch fill an SM's shared memory
}

namespace {

// Parameters shared by the bf16/fp32 and e4m3 launchers; returns the grid size.
int decode_params(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                  const int32_t *kv_indices, float sm_scale, float k_scale, float v_scale, void *o, float *lse,
                  void *workspace, DecodeParams &p) {
    const bsp_problem &P = plan->problem;
    p.ws = static_cast<const uint8_t *>(workspace);
    p.off_queue = plan->off_queue_indptr;
    p.off_items = plan->off_items;
    p.off_plse = plan->off_partial_lse;
    p.off_po = plan->off_partial_o;
    p.off_status = plan->off_status;
    p.off_merges = plan->off_merges;
    p.q = q; p.k = k_pages; p.v = v_pages;
    p.kv_indices = kv_indices;
    p.o = o;
    p.lse = lse;
    // s = sm_scale * q . (k_scale * k): the K scale folds into the score scale
    const float qk_scale = sm_scale * k_scale;
    p.scale_log2 = qk_scale * kLog2e;
    p.v_scale = v_scale;
    p.sink = P.sink;
    p.window_left = P.window_left;
    p.soft_cap_on = P.logits_soft_cap > 0.f;
    p.cap_in = p.soft_cap_on ? qk_scale / P.logits_soft_cap : 0.f;
    p.cap_out = P.logits_soft_cap * kLog2e;
    p.H_qo = P.num_qo_heads;
    p.H_kv = P.num_kv_heads;
    p.g = plan->group;
    p.page_size = P.page_size;
    p.tile_rows = plan->tile_rows;
    // A plan may have more queues than CTAs fit on the GPU at once: each CTA then
    // runs several consecutive queues (one wave; the planner balanced every queue).
    const int sms = num_sms_of_current_device(nullptr);
    if (sms < 0) return -1;
    const int resident = sms * decode_ctas_per_sm(P.head_dim, P.dtype);
    p.num_queues = plan->capacity.num_ctas;
    p.queues_per_cta = (p.num_queues + resident - 1) / resident;
    return (p.num_queues + p.queues_per_cta - 1) / p.queues_per_cta;
}

}  // namespace

int launch_decode(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                  const int32_t *kv_indices, int64_t num_pages, float sm_scale, void *o, float *lse,
                  void *workspace, cudaStream_t stream) {
    const bsp_problem &P = plan->problem;
    DecodeParams p;
    const int grid = decode_params(plan, q, k_pages, v_pages, kv_indices, sm_scale, 1.f, 1.f, o, lse, workspace, p);
    if (grid < 0) return fail(BSP_ERR_CUDA, "no current CUDA device");
    if (P.dtype == BSP_DTYPE_BF16) {
        if (p.g > kMmaRows) return fail(BSP_ERR_UNSUPPORTED, "bf16 decode needs num_qo_heads / num_kv_heads <= 16");
        if (P.head_dim != 128 && P.head_dim != 64) return fail(BSP_ERR_UNSUPPORTED, "bf16 decode supports head_dim 64 and 128");
        // Page rows are contiguous, so pages of 8 or more tokens (powers of two)
        // are gathered by TMA, one tensor copy per page box; smaller pages by
        // 16-byte cp.async. Without the pool size (num_pages 0) no map is made.
        const int ps = P.page_size;
        const bool tma = num_pages > 0 && ps >= 8 && (ps & (ps - 1)) == 0 &&
                         num_pages * (int64_t)ps <= INT32_MAX;
        CUtensorMap tk, tv;
        std::memset(&tk, 0, sizeof(tk));
        std::memset(&tv, 0, sizeof(tv));
        if (tma) {
            p.box_rows = ps < kTileK ? ps : kTileK;
            const uint64_t rows = (uint64_t)num_pages * ps;
            int rc = make_tmap_bf16(&tk, k_pages, P.head_dim, P.num_kv_heads, rows, 1, p.box_rows);
            if (rc == BSP_OK) rc = make_tmap_bf16(&tv, v_pages, P.head_dim, P.num_kv_heads, rows, 1, p.box_rows);
            if (rc != BSP_OK) return rc;
            return P.head_dim == 128 ? launch_decode_bf16<128, true>(tk, tv, p, grid, stream)
                                     : launch_decode_bf16<64, true>(tk, tv, p, grid, stream);
        }
        p.box_rows = 0;
        return P.head_dim == 128 ? launch_decode_bf16<128, false>(tk, tv, p, grid, stream)
                                 : launch_decode_bf16<64, false>(tk, tv, p, grid, stream);
    }
    switch (P.head_dim) {
        case 32: return launch_decode_f32<32>(p, grid, stream);
        case 64: return launch_decode_f32<64>(p, grid, stream);
        case 128: return launch_decode_f32<128>(p, grid, stream);
        case 256: return launch_decode_f32<256>(p, grid, stream);
        default: return fail(BSP_ERR_UNSUPPORTED, "fp32 decode supports head_dim 32, 64, 128, 256");
    }
}

int launch_decode_fp8(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *kv_indices, int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                      void *o, float *lse, void *workspace, cudaStream_t stream) {
    const bsp_problem &P = plan->problem;
    if (P.dtype != BSP_DTYPE_BF16 || P.head_dim != 128)
        return fail(BSP_ERR_UNSUPPORTED, "e4m3 KV decode needs a bf16 problem (queries, outputs) with head_dim 128");
    if (plan->group > kMmaRows) return fail(BSP_ERR_UNSUPPORTED, "e4m3 KV decode needs num_qo_heads / num_kv_heads <= 16");
    const int ps = P.page_size;
    if (ps < 8 || (ps & (ps - 1)) != 0)
        return fail(BSP_ERR_UNSUPPORTED, "e4m3 KV decode needs a power-of-two page size of at least 8");
    if (num_pages <= 0 || num_pages * (int64_t)ps > INT32_MAX)
        return fail(BSP_ERR_INVALID_ARG, "e4m3 KV decode needs the pool size: 0 < num_pages * page_size <= 2^31 - 1");
    if (!(std::isfinite(k_scale) && std::isfinite(v_scale)) || k_scale <= 0.f || v_scale <= 0.f)
        return fail(BSP_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive");
    DecodeParams p;
    const int grid = decode_params(plan, q, k_pages, v_pages, kv_indices, sm_scale, k_scale, v_scale, o, lse,
                                   workspace, p);
    if (grid < 0) return fail(BSP_ERR_CUDA, "no current CUDA device");
    p.box_rows = ps < kTileK ? ps : kTileK;
    const uint64_t rows = (uint64_t)num_pages * ps;
    CUtensorMap tk, tv;
    int rc = make_tmap(&tk, k_pages, 1, P.head_dim, P.num_kv_heads, rows, 1, p.box_rows);
    if (rc == BSP_OK) rc = make_tmap(&tv, v_pages, 1, P.head_dim, P.num_kv_heads, rows, 1, p.box_rows);
    if (rc != BSP_OK) return rc;
    return plan->group <= 8 ? launch_decode_bf16<128, true, true, 1>(tk, tv, p, grid, stream)
                            : launch_decode_bf16<128, true, true, 2>(tk, tv, p, grid, stream);
}

int launch_wait_probe(long long limit_cycles, int *status, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(limit_cycles, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("wait probe launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

int launch_reduce(const bsp_plan_info *plan, void *o, float *lse, void *workspace, cudaStream_t stream) {
    const bsp_problem &P = plan->problem;
    ReduceParams p;
    p.ws = static_cast<const uint8_t *>(workspace);
    p.off_header = plan->off_header;
    p.off_merges = plan->off_merges;
    p.off_plse = plan->off_partial_lse;
    p.off_po = plan->off_partial_o;
    p.o = o;
    p.lse = lse;
    p.H_qo = P.num_qo_heads;
    p.g = plan->group;
    p.tile_rows = plan->tile_rows;
    p.sink = P.sink;
    const bool bf = P.dtype == BSP_DTYPE_BF16;
    const int64_t u = (int64_t)plan->num_merges * plan->tile_rows * (P.head_dim / 4);
    switch (P.head_dim) {
        case 32: return bf ? launch_reduce_t<32, __nv_bfloat16>(p, u, stream) : launch_reduce_t<32, float>(p, u, stream);
        case 64: return bf ? launch_reduce_t<64, __nv_bfloat16>(p, u, stream) : launch_reduce_t<64, float>(p, u, stream);
        case 128:
            return bf ? launch_reduce_t<128, __nv_bfloat16>(p, u, stream) : launch_reduce_t<128, float>(p, u, stream);
        case 256:
            return bf ? launch_reduce_t<256, __nv_bfloat16>(p, u, stream) : launch_reduce_t<256, float>(p, u, stream);
        default: return fail(BSP_ERR_UNSUPPORTED, "head_dim must be 32, 64, 128 or 256");
    }
}

}  // namespace bsp
