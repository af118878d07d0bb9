// Ragged (causal) prefill over a paged KV cache on the tcgen05 tensor cores.
//
// What it computes (FlashInfer: Making Attention Fit the Serving Workload,
// §2.1 eq 1, §3.1 eq 4-5): for each work item of the plan — a query tile of
// 256 packed rows (positions x the g query heads of one kv head, technical
// review eq 3) and one chunk of that tile's visible KV — the attention state
// (O, LSE) over the chunk, with the bottom-right causal mask (FlashInfer 原理
// overview, ⑧). Unsplit tiles write the final output, split ones an fp32
// partial state that the reduction kernel merges (overview ⑨).
//
// How (sparse gather, dense compute: overview ⑥, engineering walkthrough
// §IV.2 and §V.4): the KV chunk is walked in tiles of 128 tokens. Rows are
// contiguous inside a page, so each page (or 128-token piece of a page) of K
// and of V is one TMA tensor copy into a 128-byte-swizzled shared-memory tile;
// the page table only supplies the copy's row coordinate. The 256 query rows
// are two 128-row MMA subtiles that share every K and V tile. One CTA per SM,
// persistent over its plan queue, ten warps:
//   warp 0      TMA: both Q subtiles of the item, then K and V tiles into two
//               2-stage rings (K is released after the second S, V after the
//               second PV)
//   warp 1      TMEM owner and MMA issuer, in the order
//               S0(0) S1(0) | PV0(t) S0(t+1) PV1(t) S1(t+1) | ...
//               S = Q K^T (M 128, N 128, K 128) into TMEM; P (bf16) is written
//               back over S in TMEM and O += P V takes P straight from TMEM
//               (V as an MN-major shared-memory operand)
//   warps 2-5   softmax of subtile 0, warps 6-9 softmax of subtile 1: one thread
//               per row; scale, mask (only on tiles that need it), base-2 online
//               softmax, P to TMEM, O rescale in TMEM, epilogue O / l and LSE.
//               O is read out of TMEM at once (freeing it for the next item's
//               PV); each warp turns its 32 bf16 output rows around in a small
//               swizzled shared-memory buffer so that its global stores cover
//               whole 128-byte lines (fp32 partial states are stored directly).
// While one softmax group works on its S, the tensor core runs the other
// subtile's PV and next S. The reference maximum of a row is only moved when
// the running maximum exceeds it by more than 8 (a factor 256): the result is
// exact because O and l always share the same reference, and O in TMEM is
// rescaled only then. MMAs of the CTA execute in issue order, so S(t+1) cannot
// overwrite P(t) before PV(t) has read it, and once S(t) is complete PV(t-1)
// is too.
// Every wait is a bounded spin (SM clock cycles); a wait that gives
// up sets the workspace status word and an abort flag, and the CTA finishes
// without further work.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "bsp_internal.h"
#include "device_common.cuh"
#include "sm100.cuh"

namespace bsp {
namespace {

using namespace sm100;

constexpr int kSub = 2;           // 128-row subtiles per query tile
constexpr int kRows = 128;        // rows per subtile (M)
constexpr int kKvTile = 128;      // KV tokens per tile
constexpr int kD = 128;           // head dim
constexpr int kThreads = 320;     // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
// the cp.async gather adds warp 10: warp 0 copies K, warp 10 V (one warp alone
// cannot keep enough 16-byte copies in flight)
constexpr int kThreadsGather = 352;
constexpr int kVWarp = 10;
constexpr int kHalf = 16384;      // [128 rows][64 bf16], 128-byte swizzle
constexpr int kTile = 2 * kHalf;  // [128 rows][128 bf16]

constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kOffQ = 0;                          // kSub tiles
constexpr int kOffK = kOffQ + kSub * kTile;       // kKStages tiles
constexpr int kOffV = kOffK + kKStages * kTile;   // kVStages tiles
constexpr int kStgWarp = 32 * 128;                 // per softmax warp: 32 rows x 64 bf16, swizzled
constexpr int kOffStg = kOffV + kVStages * kTile;  // output staging, 8 warps
constexpr int kOffBar = kOffStg + 8 * kStgWarp;
// Ring barriers are indexed kKFull0 + stage etc.: one slot per stage of each ring.
enum Bar {
    kQFull = 0, kQEmpty,
    kKFull0, kKEmpty0 = kKFull0 + kKStages, kVFull0 = kKEmpty0 + kKStages, kVEmpty0 = kVFull0 + kVStages,
    kSFull0 = kVEmpty0 + kVStages, kSFull1, kPFull0, kPFull1, kODone0, kODone1, kOFree0, kOFree1, kNumBars
};
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 227 * 1024, "prefill tiles exceed shared memory");

// TMEM columns: S0 (P0 over its first 64 columns) | S1 (P1) | O0 | O1
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s at 2 GHz: a fault, not a stall
constexpr int kStatusWait = 0x201;
constexpr float kRescaleThreshold = 8.f;  // log2 units

struct PrefillParams {
    const uint8_t *ws;
    uint64_t off_queue, off_items, off_plse, off_po, off_status;
    const int32_t *kv_indices;
    const char *k, *v;  // page pools (cp.async gather)
    void *o;
    float *lse;
    float scale_log2;
    int H_qo, H_kv, g, page_size, box_rows, causal, tile_rows;
    int queues_per_cta, num_queues;  // CTA b runs plan queues [b * qpc, min((b + 1) * qpc, C))
    int contig;              // K / V tensor maps cover the gather region: request b's token t is row
                             // page_base * page_size + t (boxes of 128 rows, no page lookup)
    int window_left;         // > 0: key j is masked for a row at position i if j < i + kv_len - qo_len - window_left
    int soft_cap_on;         // scores become tanh(s * cap_in); scale_log2 is then c * log2(e)
    float cap_in;            // sm_scale / c
    const float *sink;       // per-qo-head sink logits, or null (applied to finished rows)
};

struct Ctx {
    volatile int *abort_flag;
    int *status;
};

__device__ __forceinline__ bool wait_bar(const Ctx &c, uint32_t bar, uint32_t parity) {
    if (mbar_wait_spin(bar, parity, kWaitLimitCycles, c.abort_flag)) return true;
    *c.abort_flag = 1;
    atomicCAS(c.status, 0, kStatusWait);
    return false;
}
// Same, with one outcome for the whole warp.
__device__ __forceinline__ bool wait_bar_warp(const Ctx &c, uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_bar(c, bar, parity));
}

// Paired fp32 arithmetic (one instruction for two elements).
__device__ __forceinline__ void fma2_bcast(float &d0, float &d1, float a0, float a1, float b, float c) {
    asm("{ .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n mov.b64 rc, {%5, %5};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1) {
    asm("{ .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n add.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d0), "=f"(d1)
        : "f"(d0), "f"(d1), "f"(a0), "f"(a1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}

// A read-only global load issued where it stands (its value is waited for at first use).
__device__ __forceinline__ int ld_nc_s32(const int *p) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// kTma: K and V tiles arrive by TMA tensor copies, one per page box (pages of
// 8 or more tokens); otherwise by 16-byte cp.async copies written straight into
// the same 128-byte-swizzled layout (pages of any size, e.g. 1).
// kVar: the sliding window and logits soft-cap variants are compiled in (the
// default instantiation has neither, at no cost).
template <bool kTma, bool kVar>
__global__ void __launch_bounds__(kTma ? kThreads : kThreadsGather, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = dev::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t *queue = reinterpret_cast<const int32_t *>(p.ws + p.off_queue);
    const bsp_work_item *items = reinterpret_cast<const bsp_work_item *>(p.ws + p.off_items);
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the merge kernel may get resident now
    const int qb = blockIdx.x * p.queues_per_cta;
    const int it0 = queue[qb], it1 = queue[min(qb + p.queues_per_cta, p.num_queues)];
    if (it0 >= it1) return;  // uniform across the CTA, before any barrier

    auto bar = [&](int i) { return sb + kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);
    Ctx ctx{reinterpret_cast<volatile int *>(smem + kOffAbort),
            reinterpret_cast<int *>(const_cast<uint8_t *>(p.ws) + p.off_status)};

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool softmax_arrivals = i == kPFull0 || i == kPFull1 || i == kOFree0 || i == kOFree1;
            const bool kv_full = (i >= kKFull0 && i < kKFull0 + kKStages) || (i >= kVFull0 && i < kVFull0 + kVStages);
            mbar_init(bar(i), softmax_arrivals ? 128 : (kv_full && !kTma) ? 32 : 1);  // cp.async: one per lane
        }
        *ctx.abort_flag = 0;
        fence_barrier_init();
    }
    // V ring starts zeroed: rows a tile does not copy then always hold finite values
    for (int i = threadIdx.x; i < kVStages * kTile / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem + kOffV)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 1) {
        tmem_alloc(dev::smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int g = p.g;
    const int pos_per_sub = kRows / g;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        int q_cnt = 0, j = 0;  // j: KV tiles issued so far
        bool ok = true;
        for (int it = it0; it < it1 && ok; ++it) {
            const bsp_work_item w = items[it];
            const int len = w.kv_end - w.kv_start;
            const int nt = (len + kKvTile - 1) / kKvTile;
            if (nt == 0) continue;
            if (!(ok = wait_bar_warp(ctx, bar(kQEmpty), (q_cnt & 1) ^ 1))) break;
            ++q_cnt;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(kQFull), kSub * kTile);
#pragma unroll
                for (int sub = 0; sub < kSub; ++sub)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sb + kOffQ + sub * kTile + h * kHalf, &tq, bar(kQFull), h * 64, w.kv_head * g,
                                    w.q_tok0 + sub * pos_per_sub);
            }
            int pg_next[kKvTile / 32];  // cp.async gather: page ids of this lane's keys in the next tile
            auto lookup = [&](int (&pg)[kKvTile / 32], int tt) {
#pragma unroll
                for (int i = 0; i < kKvTile / 32; ++i) {
                    const int key = tt * kKvTile + lane + 32 * i;
                    pg[i] = key < len ? __ldg(p.kv_indices + w.page_base + (w.kv_start + key) / p.page_size) : 0;
                }
            };
            (void)lookup;
            for (int t = 0; t < nt; ++t, ++j) {
                const int tok0 = w.kv_start + t * kKvTile;
                const int valid = min(kKvTile, len - t * kKvTile);
                const int stage = j % kKStages, round = j / kKStages;
                const int vst = j % kVStages, vrd = j / kVStages;
                if constexpr (kTma) {
                    const int nseg = (valid + p.box_rows - 1) / p.box_rows;
                    int row0;
                    if (p.contig) {
                        row0 = w.page_base * p.page_size + tok0 + lane * p.box_rows;
                    } else {
                        int page = 0;
                        if (lane < nseg)
                            page = __ldg(p.kv_indices + w.page_base + (tok0 + lane * p.box_rows) / p.page_size);
                        row0 = page * p.page_size + (tok0 + lane * p.box_rows) % p.page_size;
                    }
                    const uint32_t seg = (uint32_t)lane * p.box_rows * 128;
                    const uint32_t bytes = (uint32_t)nseg * p.box_rows * 128 * 2;
                    if (!(ok = wait_bar_warp(ctx, bar(kKEmpty0 + stage), (round & 1) ^ 1))) break;
                    if (lane == 0) mbar_arrive_expect_tx(bar(kKFull0 + stage), bytes);
                    __syncwarp();
                    if (lane < nseg) {
                        const uint32_t d = sb + kOffK + stage * kTile + seg;
                        tma_load_3d(d, &tk, bar(kKFull0 + stage), 0, w.kv_head, row0);
                        tma_load_3d(d + kHalf, &tk, bar(kKFull0 + stage), 64, w.kv_head, row0);
                    }
                    if (!(ok = wait_bar_warp(ctx, bar(kVEmpty0 + vst), (vrd & 1) ^ 1))) break;
                    if (lane == 0) mbar_arrive_expect_tx(bar(kVFull0 + vst), bytes);
                    __syncwarp();
                    if (lane < nseg) {
                        const uint32_t d = sb + kOffV + vst * kTile + seg;
                        tma_load_3d(d, &tv, bar(kVFull0 + vst), 0, w.kv_head, row0);
                        tma_load_3d(d + kHalf, &tv, bar(kVFull0 + vst), 64, w.kv_head, row0);
                    }
                } else {
                    // Lane l looks up keys l + 32 i (page ids read one tile ahead); each
                    // warp instruction then copies the sixteen 16-byte chunks of two keys
                    // into their swizzled places. Keys past the chunk end are not copied
                    // (their rows keep finite values).
                    uint64_t off[kKvTile / 32];
                    if (t == 0) lookup(pg_next, 0);
#pragma unroll
                    for (int i = 0; i < kKvTile / 32; ++i) {
                        const int key = lane + 32 * i;
                        const int tk_ = tok0 + key;
                        off[i] = key < valid ? (((uint64_t)pg_next[i] * p.page_size + tk_ % p.page_size) * p.H_kv +
                                                w.kv_head) * (kD * 2)
                                             : 0;
                    }
                    if (t + 1 < nt) lookup(pg_next, t + 1);
                    auto copy_tile = [&](const char *src, uint32_t dst, uint32_t full) {
                        const int c = lane & 15;
#pragma unroll
                        for (int ii = 0; ii < kKvTile / 2; ++ii) {
                            const int key = 2 * ii + (lane >> 4);  // key >> 5 == ii >> 4 for the whole warp
                            const uint64_t o = __shfl_sync(0xffffffffu, off[ii >> 4], key & 31);
                            if (key < valid)
                                dev::cp_async_16(dst + (c >> 3) * kHalf + key * 128 + (((c & 7) ^ (key & 7)) << 4),
                                                 src + o + c * 16, 16);
                        }
                        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(full) : "memory");
                    };
                    (void)vst;
                    (void)vrd;
                    if (!(ok = wait_bar_warp(ctx, bar(kKEmpty0 + stage), (round & 1) ^ 1))) break;
                    copy_tile(p.k, sb + kOffK + stage * kTile, bar(kKFull0 + stage));  // V: warp kVWarp
                }
            }
        }
        if constexpr (!kTma) asm volatile("cp.async.wait_all;\n" ::: "memory");  // nothing in flight at exit
    } else if (!kTma && warp == kVWarp) {
        // ------------------------------------------------ V gather (cp.async)
        // The same items and tiles as warp 0, V rows only: lane l looks up keys
        // l + 32 i one tile ahead, each warp instruction copies two keys' sixteen
        // 16-byte chunks into their swizzled places.
        int j = 0;
        bool ok = true;
        for (int it = it0; it < it1 && ok; ++it) {
            const bsp_work_item w = items[it];
            const int len = w.kv_end - w.kv_start;
            const int nt = (len + kKvTile - 1) / kKvTile;
            int pg_next[kKvTile / 32];
            auto lookup = [&](int (&pg)[kKvTile / 32], int tt) {
#pragma unroll
                for (int i = 0; i < kKvTile / 32; ++i) {
                    const int key = tt * kKvTile + lane + 32 * i;
                    pg[i] = key < len ? __ldg(p.kv_indices + w.page_base + (w.kv_start + key) / p.page_size) : 0;
                }
            };
            if (nt > 0) lookup(pg_next, 0);
            for (int t = 0; t < nt; ++t, ++j) {
                const int tok0 = w.kv_start + t * kKvTile;
                const int valid = min(kKvTile, len - t * kKvTile);
                const int vst = j % kVStages, vrd = j / kVStages;
                uint64_t off[kKvTile / 32];
#pragma unroll
                for (int i = 0; i < kKvTile / 32; ++i) {
                    const int key = lane + 32 * i;
                    const int tk_ = tok0 + key;
                    off[i] = key < valid ? (((uint64_t)pg_next[i] * p.page_size + tk_ % p.page_size) * p.H_kv +
                                            w.kv_head) * (kD * 2)
                                         : 0;
                }
                if (t + 1 < nt) lookup(pg_next, t + 1);
                if (!(ok = wait_bar_warp(ctx, bar(kVEmpty0 + vst), (vrd & 1) ^ 1))) break;
                const uint32_t dst = sb + kOffV + vst * kTile;
                const char *src = p.v;
                const int c = lane & 15;
#pragma unroll
                for (int ii = 0; ii < kKvTile / 2; ++ii) {
                    const int key = 2 * ii + (lane >> 4);  // key >> 5 == ii >> 4 for the whole warp
                    const uint64_t o = __shfl_sync(0xffffffffu, off[ii >> 4], key & 31);
                    if (key < valid)
                        dev::cp_async_16(dst + (c >> 3) * kHalf + key * 128 + (((c & 7) ^ (key & 7)) << 4),
                                         src + o + c * 16, 16);
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar(kVFull0 + vst))
                             : "memory");
            }
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");  // nothing in flight at exit
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // One thread issues everything: between MMA groups the tensor pipe
        // drains, so every cycle spent on warp votes, redundant fences or index
        // arithmetic here is idle tensor time. The only fence needed is after
        // the P barrier (P arrives through tcgen05.st from other threads); K, V
        // and Q arrive through TMA (async proxy) with their mbarriers.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kRows, kKvTile, false, false);
            constexpr uint32_t id_pv = idesc_bf16_f32(kRows, kD, false, true);
            int q_cnt = 0, p_cnt0 = 0, p_cnt1 = 0, done = 0;
            int kst = 0, kph = 0;  // K ring position of the next tile: stage, phase
            int vst = 0, vph = 0;  // V ring position of the next tile
            bool ok = true;
            auto wait1 = [&](uint32_t b, uint32_t parity) -> bool {
                if (mbar_wait_spin(b, parity, kWaitLimitCycles, ctx.abort_flag)) return true;
                *ctx.abort_flag = 1;
                atomicCAS(ctx.status, 0, kStatusWait);
                return false;
            };
            auto issue_s = [&](int sub, int stage) {
                const uint32_t sq = sb + kOffQ + sub * kTile, sk = sb + kOffK + stage * kTile;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16_ss(tmem + sub * 128, smem_desc_sw128(sq + o, 16, 1024), smem_desc_sw128(sk + o, 16, 1024),
                                id_s, kk > 0);
                }
                mma_commit(bar(kSFull0 + sub));
            };
            auto issue_pv = [&](int sub, int stage, bool acc) {
                const uint32_t sv = sb + kOffV + stage * kTile;
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk)
                    mma_bf16_ts(tmem + 256 + sub * 128, tmem + sub * 128 + kk * 8,
                                smem_desc_sw128(sv + kk * 16 * 128, kHalf, 1024), id_pv, acc || kk > 0);
            };
            // the next item's KV range is read one item ahead (its latency then
            // overlaps this item's MMAs instead of delaying the next item's first S)
            int nt_next = (items[it0].kv_end - items[it0].kv_start + kKvTile - 1) / kKvTile;
            for (int it = it0; it < it1 && ok; ++it) {
                const int nt = nt_next;
                int ks = 0, ke = 0;
                if (it + 1 < it1) {
                    ks = ld_nc_s32(&items[it + 1].kv_start);
                    ke = ld_nc_s32(&items[it + 1].kv_end);
                }
                if (nt == 0) {
                    nt_next = (ke - ks + kKvTile - 1) / kKvTile;
                    continue;
                }
                if (!(ok = wait1(bar(kQFull), q_cnt & 1))) break;
                ++q_cnt;
                // prologue: S0(0), S1(0) on K tile 0 of the item
                if (!(ok = wait1(bar(kKFull0 + kst), kph))) break;
                issue_s(0, kst);
                issue_s(1, kst);
                mma_commit(bar(kKEmpty0 + kst));
                if (nt == 1) mma_commit(bar(kQEmpty));
                if (++kst == kKStages) { kst = 0; kph ^= 1; }
                for (int t = 0; t < nt && ok; ++t) {
                    if (!(ok = wait1(bar(kVFull0 + vst), vph))) break;
                    const bool more = t + 1 < nt;
                    // subtile 0: PV0(t), S0(t+1)
                    if (!(ok = wait1(bar(kPFull0), p_cnt0 & 1))) break;
                    ++p_cnt0;
                    if (t == 0 && done > 0 && !(ok = wait1(bar(kOFree0), (done - 1) & 1))) break;
                    tc_fence_after();
                    issue_pv(0, vst, t > 0);
                    if (!more) mma_commit(bar(kODone0));
                    if (more) {
                        if (!(ok = wait1(bar(kKFull0 + kst), kph))) break;
                        issue_s(0, kst);
                    }
                    // subtile 1: PV1(t), S1(t+1)
                    if (!(ok = wait1(bar(kPFull1), p_cnt1 & 1))) break;
                    ++p_cnt1;
                    if (t == 0 && done > 0 && !(ok = wait1(bar(kOFree1), (done - 1) & 1))) break;
                    tc_fence_after();
                    issue_pv(1, vst, t > 0);
                    if (!more) mma_commit(bar(kODone1));
                    mma_commit(bar(kVEmpty0 + vst));
                    if (++vst == kVStages) { vst = 0; vph ^= 1; }
                    if (more) {
                        issue_s(1, kst);
                        mma_commit(bar(kKEmpty0 + kst));
                        if (t + 1 == nt - 1) mma_commit(bar(kQEmpty));
                        if (++kst == kKStages) { kst = 0; kph ^= 1; }
                    }
                }
                ++done;
                nt_next = (ke - ks + kKvTile - 1) / kKvTile;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int sub = (warp - 2) >> 2;       // warps 2-5: subtile 0, warps 6-9: subtile 1
        const int q4 = warp & 3;               // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;          // row within the subtile
        const int rt = sub * kRows + r;        // row within the 256-row tile
        const uint32_t tl = (uint32_t)(q4 * 32) << 16;
        const uint32_t tS = tmem + tl + sub * 128, tO = tmem + tl + 256 + sub * 128;
        float *plse = reinterpret_cast<float *>(const_cast<uint8_t *>(p.ws) + p.off_plse);
        float *po = reinterpret_cast<float *>(const_cast<uint8_t *>(p.ws) + p.off_po);
        int s_cnt = 0, o_cnt = 0, j = 0;
        bool ok = true;
        for (int it = it0; it < it1 && ok; ++it) {
            const bsp_work_item w = items[it];
            const int len = w.kv_end - w.kv_start;
            const int nt = (len + kKvTile - 1) / kKvTile;
            const int pos = w.pos0 + rt / g;
            const int lo = kVar && p.window_left > 0 ? pos + w.kv_len - w.qo_len - p.window_left : INT_MIN;  // window edge
            const int lim = p.causal ? pos + w.kv_len - w.qo_len : INT_MAX;  // key j allowed iff j <= lim
            asm volatile("" ::"r"(lim), "r"(len), "r"(w.kv_start));  // loaded before the S wait, not after
            float m = -INFINITY, l = 0.f;  // m: reference maximum (scaled, base 2)
            for (int t = 0; t < nt; ++t, ++j) {
                const int tok0 = w.kv_start + t * kKvTile;
                const int valid = min(kKvTile, len - t * kKvTile);
                if (!(ok = wait_bar_warp(ctx, bar(kSFull0 + sub), s_cnt & 1))) break;
                ++s_cnt;
                tc_fence_after();
                float sv[kKvTile];
#pragma unroll
                for (int c = 0; c < kKvTile / 32; ++c) {
                    float v[32];
                    tmem_ld32(tS + c * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sv[c * 32 + i] = v[i];
                }
                tmem_wait_ld();
                if (kVar && p.soft_cap_on) {  // technical review eq 8 (c * tanh(s / c), the factor c folded into scale_log2)
#pragma unroll
                    for (int c = 0; c < kKvTile; ++c) sv[c] = dev::tanh_ex2(sv[c] * p.cap_in);
                }
                const bool full = valid == kKvTile && tok0 + kKvTile - 1 <= lim && tok0 >= lo;
                if (!full) {
                    // visible columns of this row: [c_lo, c_hi)
                    const int c_hi = min(valid, lim == INT_MAX ? kKvTile : max(0, min(kKvTile, lim - tok0 + 1)));
                    const int c_lo = kVar && lo != INT_MIN ? max(0, lo - tok0) : 0;
                    // a late row's window can start past this KV tile (a 256-row tile
                    // spans 128+ positions when g <= 2): nothing visible then
                    const int c_w = max(0, c_hi - c_lo);
                    if (kVar) {
#pragma unroll
                        for (int c = 0; c < kKvTile; ++c)
                            sv[c] = (unsigned)(c - c_lo) < (unsigned)c_w ? sv[c] : -INFINITY;
                    } else {
#pragma unroll
                        for (int c = 0; c < kKvTile; ++c) sv[c] = c < c_hi ? sv[c] : -INFINITY;
                    }
                }
                // row maximum: 8 independent chains of 3-input maxima
                float pm[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) pm[i] = fmaxf(sv[2 * i], sv[2 * i + 1]);
#pragma unroll
                for (int c = 16; c < kKvTile; c += 2) pm[(c >> 1) & 7] = max3(pm[(c >> 1) & 7], sv[c], sv[c + 1]);
                const float mx = max3(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
                const float mxs = mx * p.scale_log2;                 // scale > 0 keeps the order
                const bool move = mxs > m + kRescaleThreshold;       // false for an all-masked row
                const float alpha = move ? ex2(m - mxs) : 1.f;       // 0 when m was -inf
                if (move) {
                    l *= alpha;
                    m = mxs;
                }
                const float ref = m == -INFINITY ? 0.f : m;
                float ps[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ps[i] = 0.f;
#pragma unroll
                for (int c = 0; c < kKvTile; c += 2) {
                    fma2_bcast(sv[c], sv[c + 1], sv[c], sv[c + 1], p.scale_log2, -ref);
                    sv[c] = ex2(sv[c]);
                    sv[c + 1] = ex2(sv[c + 1]);
                    const int a = (c >> 1) & 3;
                    add2(ps[2 * a], ps[2 * a + 1], sv[c], sv[c + 1]);
                }
                l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                // P (bf16 pairs) over the first 64 columns of S
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) pk[i] = dev::pack_bf16(sv[c * 64 + 2 * i], sv[c * 64 + 2 * i + 1]);
                    tmem_st32_u(tS + c * 32, pk);
                }
                // O rescale when the reference moved (PV(t-1) is complete: S(t) is)
                if (t > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        float v[32];
                        tmem_ld32(tO + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= alpha;
                        tmem_st32(tO + c * 32, v);
                    }
                }
                tmem_wait_st();
                const int vz_end = min(kKvTile, (valid + p.box_rows - 1) / p.box_rows * p.box_rows);
                if (sub == 0 && valid < vz_end) {
                    // rows of the last copied box past the chunk end may hold anything:
                    // zero them so that P = 0 meets finite values (rows past the box keep
                    // an earlier tile's finite values, the ring starts zeroed)
                    const int vst = j % kVStages, vrd = j / kVStages;
                    if (!(ok = wait_bar_warp(ctx, bar(kVFull0 + vst), vrd & 1))) break;
                    if (r >= valid && r < vz_end) {
                        uint4 *v0 = reinterpret_cast<uint4 *>(smem + kOffV + vst * kTile + r * 128);
                        uint4 *v1 = reinterpret_cast<uint4 *>(smem + kOffV + vst * kTile + kHalf + r * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) v0[i] = v1[i] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(bar(kPFull0 + sub));
            }
            if (!ok) break;
            // ---- epilogue: O / l, LSE; final output or partial state ----
            // O leaves TMEM first, so that the next item's PV may start while
            // this one is written out.
            float ov[kD];
            if (nt > 0) {
                if (!(ok = wait_bar_warp(ctx, bar(kODone0 + sub), o_cnt & 1))) break;
                ++o_cnt;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    float v[32];
                    tmem_ld32(tO + c * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[c * 32 + i] = v[i];
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(kOFree0 + sub));
            } else {
#pragma unroll
                for (int i = 0; i < kD; ++i) ov[i] = 0.f;
            }
            const bool has = l > 0.f;
            float inv = has ? 1.f / l : 0.f;
            float lse_v = has ? (m + log2f(l)) * dev::kLn2 : -INFINITY;
            const size_t orow = (size_t)(w.q_tok0 + rt / g) * p.H_qo + (size_t)w.kv_head * g + (rt % g);
            const size_t prow = (size_t)w.slot * p.tile_rows + rt;
            const int n_rows = w.n_pos * g;  // real rows of the tile
            if (p.sink && w.slot < 0 && rt < n_rows) inv *= dev::fold_sink(lse_v, p.sink[w.kv_head * g + rt % g]);
            if (w.slot < 0) {
                // bf16 output through this warp's swizzled staging, 64 columns at a
                // time: each thread writes its row, then every store instruction
                // covers four whole 128-byte lines (lane l: row 4i + l/8, chunk l%8)
                const uint32_t stg = sb + kOffStg + (warp - 2) * kStgWarp;
                const int cc = lane & 7;
                const int rt_base = sub * kRows + q4 * 32;
                unsigned long long orr[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) orr[i] = __shfl_sync(0xffffffffu, (unsigned long long)orow, 4 * i + (lane >> 3));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float *x = ov + h * 64 + q * 8;
                        st_shared_v4(stg + lane * 128 + ((q ^ (lane & 7)) << 4), dev::pack_bf16(x[0] * inv, x[1] * inv),
                                     dev::pack_bf16(x[2] * inv, x[3] * inv), dev::pack_bf16(x[4] * inv, x[5] * inv),
                                     dev::pack_bf16(x[6] * inv, x[7] * inv));
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3);
                        const uint4 val = ld_shared_v4(stg + rr * 128 + ((cc ^ (rr & 7)) << 4));
                        if (rt_base + rr < n_rows)
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + orr[i] * kD + h * 64 + cc * 8) =
                                val;
                    }
                    __syncwarp();
                }
            } else if (rt < n_rows) {
                // fp32 partial state: this thread's row is 512 contiguous bytes
                float4 *dst = reinterpret_cast<float4 *>(po + prow * kD);
#pragma unroll
                for (int q = 0; q < kD / 4; ++q)
                    dst[q] = make_float4(ov[q * 4] * inv, ov[q * 4 + 1] * inv, ov[q * 4 + 2] * inv, ov[q * 4 + 3] * inv);
            }
            if (rt < n_rows) {
                if (w.slot < 0) {
                    if (p.lse) p.lse[orow] = lse_v;
                } else {
                    plse[prow] = lse_v;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*ctx.abort_flag) {
        // let copies and MMAs already in flight finish before TMEM is released
        for (int i = 0; i < 100; ++i) __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Copy of the page table's pages into the gather region, in table order: one
// warp per page (grid-stride), its id read once, then the page's K and V as
// 16-byte vectors with 8 loads per lane in flight. HBM-bound: one read and one
// write of every table page.
constexpr int kStatusGatherIndex = 0x301;

__global__ void __launch_bounds__(256) gather_pages_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           uint4 *__restrict__ gk, uint4 *__restrict__ gv,
                                                           const int32_t *__restrict__ idx, int n_pages,
                                                           long long num_pages, int page_vecs, int *status) {
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long pg = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; pg < n_pages; pg += nwarps) {
        const int id = __ldg(idx + pg);
        const bool ok = id >= 0 && id < num_pages;
        if (!ok && lane == 0) atomicCAS(status, 0, kStatusGatherIndex);
        const uint4 *sk = k + (ok ? (long long)id * page_vecs : 0), *sv = v + (ok ? (long long)id * page_vecs : 0);
        uint4 *dk = gk + pg * page_vecs, *dv = gv + pg * page_vecs;
        for (int base = 0; base < page_vecs; base += 4 * 32) {
            uint4 a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + i * 32 + lane;
                a[i] = b[i] = make_uint4(0, 0, 0, 0);
                if (ok && e < page_vecs) {
                    a[i] = __ldg(sk + e);
                    b[i] = __ldg(sv + e);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + i * 32 + lane;
                if (e < page_vecs) {
                    dk[e] = a[i];
                    dv[e] = b[i];
                }
            }
        }
    }
}

}  // namespace

int launch_gather_pages(const bsp_plan_info *plan, const void *k_pages, const void *v_pages,
                        const int32_t *kv_indices, int64_t num_pages, void *workspace, cudaStream_t stream) {
    const bsp_problem &P = plan->problem;
    const int n = plan->num_table_pages;
    if (n <= 0) return BSP_OK;
    if (!kv_indices) return fail(BSP_ERR_INVALID_ARG, "kv_indices is NULL but the page table has pages");
    if (!plan->off_gather || n > plan->capacity.max_gather_pages)
        return fail(BSP_ERR_CAPACITY, "page table exceeds capacity.max_gather_pages");
    const int64_t page_bytes = (int64_t)P.page_size * P.num_kv_heads * P.head_dim * (P.dtype == BSP_DTYPE_BF16 ? 2 : 4);
    if (page_bytes % 16 != 0 || reinterpret_cast<uintptr_t>(k_pages) % 16 || reinterpret_cast<uintptr_t>(v_pages) % 16)
        return fail(BSP_ERR_INVALID_ARG, "page pools must be 16-byte aligned for the gather");
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(BSP_ERR_CUDA, "no current CUDA device");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t blocks = std::min<int64_t>((n + 7) / 8, (int64_t)sms * 16);
    gather_pages_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(k_pages), static_cast<const uint4 *>(v_pages),
        reinterpret_cast<uint4 *>(ws + plan->off_gather), reinterpret_cast<uint4 *>(ws + plan->off_gather + plan->gather_pool_bytes),
        kv_indices, n, (long long)num_pages, (int)(page_bytes / 16), reinterpret_cast<int *>(ws + plan->off_status));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("gather launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

int launch_prefill(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                   const int32_t *kv_indices, int64_t num_pages, float sm_scale, void *o, float *lse,
                   void *workspace, cudaStream_t stream) {
    const bsp_problem &P = plan->problem;
    const int g = plan->group;
    if (P.dtype != BSP_DTYPE_BF16) return fail(BSP_ERR_UNSUPPORTED, "prefill supports bf16 only");
    if (P.head_dim != kD) return fail(BSP_ERR_UNSUPPORTED, "prefill supports head_dim 128 only");
    if (plan->tile_rows != kSub * kRows || kRows % g != 0)
        return fail(BSP_ERR_UNSUPPORTED, "prefill needs 256-row tiles and 128 % g == 0");
    // Pages of 8 or more tokens (powers of two) are gathered by TMA, one tensor
    // copy per page box. Other page sizes: when the workspace has a gather
    // region that holds the page table, the pages are first copied into it in
    // table order, and every request's keys are then one contiguous run of
    // rows read by 128-row TMA boxes; otherwise 16-byte cp.async copies.
    const int ps = P.page_size;
    const bool direct = ps >= 8 && (ps & (ps - 1)) == 0 && num_pages * (int64_t)ps <= INT32_MAX;
    const bool gather = !direct && plan->off_gather != 0 && plan->num_table_pages <= plan->capacity.max_gather_pages;
    const bool tma = direct || gather;

    CUtensorMap tq, tk, tv;
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    const int box_rows = gather ? kKvTile : tma ? (ps < kKvTile ? ps : kKvTile) : 1;
    int rc = make_tmap_bf16(&tq, q, kD, P.num_qo_heads, (uint64_t)(plan->num_qo_tokens > 0 ? plan->num_qo_tokens : 1), g,
                      kRows / g);
    if (gather) {
        const uint8_t *region = static_cast<const uint8_t *>(workspace) + plan->off_gather;
        const uint64_t rows = (uint64_t)plan->capacity.max_gather_pages * ps;
        if (rc == BSP_OK) rc = make_tmap_bf16(&tk, region, kD, P.num_kv_heads, rows, 1, box_rows);
        if (rc == BSP_OK) rc = make_tmap_bf16(&tv, region + plan->gather_pool_bytes, kD, P.num_kv_heads, rows, 1, box_rows);
        if (rc == BSP_OK) rc = launch_gather_pages(plan, k_pages, v_pages, kv_indices, num_pages, workspace, stream);
    } else if (tma) {
        if (rc == BSP_OK) rc = make_tmap_bf16(&tk, k_pages, kD, P.num_kv_heads, (uint64_t)num_pages * ps, 1, box_rows);
        if (rc == BSP_OK) rc = make_tmap_bf16(&tv, v_pages, kD, P.num_kv_heads, (uint64_t)num_pages * ps, 1, box_rows);
    }
    if (rc != BSP_OK) return rc;

    PrefillParams p;
    p.ws = static_cast<const uint8_t *>(workspace);
    p.off_queue = plan->off_queue_indptr;
    p.off_items = plan->off_items;
    p.off_plse = plan->off_partial_lse;
    p.off_po = plan->off_partial_o;
    p.off_status = plan->off_status;
    p.kv_indices = kv_indices;
    p.k = static_cast<const char *>(k_pages);
    p.v = static_cast<const char *>(v_pages);
    p.H_kv = P.num_kv_heads;
    p.o = o;
    p.lse = lse;
    p.scale_log2 = sm_scale * dev::kLog2e;
    p.window_left = P.window_left;
    p.soft_cap_on = P.logits_soft_cap > 0.f;
    p.cap_in = p.soft_cap_on ? sm_scale / P.logits_soft_cap : 0.f;
    p.sink = P.sink;
    if (p.soft_cap_on) p.scale_log2 = P.logits_soft_cap * dev::kLog2e;
    p.H_qo = P.num_qo_heads;
    p.g = g;
    p.page_size = P.page_size;
    p.box_rows = box_rows;
    p.contig = gather ? 1 : 0;
    p.causal = P.causal;
    p.tile_rows = plan->tile_rows;

    static bool configured[4][64] = {{false}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(BSP_ERR_CUDA, "no current CUDA device");
    const bool var = P.window_left > 0 || P.logits_soft_cap > 0.f;
    auto kern = tma ? (var ? prefill_kernel<true, true> : prefill_kernel<true, false>)
                    : (var ? prefill_kernel<false, true> : prefill_kernel<false, false>);
    const int which = (tma ? 2 : 0) + (var ? 1 : 0);
    if (!configured[which][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("prefill smem attribute: ") + cudaGetErrorString(e));
        configured[which][dev] = true;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return fail(BSP_ERR_CUDA, "no current CUDA device");
    // more plan queues than SMs: each CTA runs several consecutive queues (one wave)
    p.num_queues = plan->capacity.num_ctas;
    p.queues_per_cta = (p.num_queues + sms - 1) / sms;
    const int grid = (p.num_queues + p.queues_per_cta - 1) / p.queues_per_cta;
    kern<<<grid, tma ? kThreads : kThreadsGather, kSmemBytes, stream>>>(tq, tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("prefill launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

}  // namespace bsp
