// merge_state: element-wise merge of two sets of attention states
// (FlashInfer: Making Attention Fit the Serving Workload, §3.2 eq 6 and §3.3
// Algorithm 1; FlashInfer 原理 overview, ④). Used to combine a shared-prefix
// view's states with the suffix view's states (walkthrough §IV.6).
//
// HBM-bound: one warp per (row, head) state; lane l holds the D/32 consecutive
// elements l*D/32 .. of the row and moves them with one vector load or store
// each (8 bytes for bf16 at D = 128, 16 for fp32) when the four O pointers are
// aligned to that size, element by element otherwise; a grid-stride loop over a
// grid sized to the SM count.
#include "bsp_internal.h"
#include "device_common.cuh"

namespace bsp {
namespace {

using namespace dev;

// E consecutive elements moved as one vector access
template <typename T, int E>
struct alignas(sizeof(T) * E) Vec {
    T v[E];
};

template <int D, typename T, bool kVec>
__global__ void __launch_bounds__(256) merge_state_kernel(const T *oa, const float *la,
                                                          const T *ob, const float *lb,
                                                          T *oo, float *lo, int64_t n) {
    constexpr int E = D / 32;
    using V = Vec<T, E>;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t s = gw; s < n; s += nw) {
        const float a = la[s], b = lb[s];
        float xa[E], xb[E];
        if constexpr (kVec) {
            const V va_ = *reinterpret_cast<const V *>(oa + s * D + lane * E);
            const V vb_ = *reinterpret_cast<const V *>(ob + s * D + lane * E);
#pragma unroll
            for (int i = 0; i < E; ++i) {
                xa[i] = to_float<T>(va_.v[i]);
                xb[i] = to_float<T>(vb_.v[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) {
                xa[i] = to_float<T>(oa[s * D + lane * E + i]);
                xb[i] = to_float<T>(ob[s * D + lane * E + i]);
            }
        }
        __syncwarp();  // every lane has read its inputs before any lane writes (in-place use)
        const bool va = a != -INFINITY, vb = b != -INFINITY;
        float wa, wb, lse;
        if (va && vb) {
            const float m = fmaxf(a, b);
            wa = exp2f((a - m) * kLog2e);
            wb = exp2f((b - m) * kLog2e);
            const float inv = 1.f / (wa + wb);
            lse = m + logf(wa + wb);
            wa *= inv;
            wb *= inv;
        } else if (va) {
            wa = 1.f; wb = 0.f; lse = a;
        } else if (vb) {
            wa = 0.f; wb = 1.f; lse = b;
        } else {
            wa = 0.f; wb = 0.f; lse = -INFINITY;
        }
        V r;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            // a pass-through side is copied exactly, never multiplied
            const float v = !vb ? (va ? xa[i] : 0.f) : !va ? xb[i] : wa * xa[i] + wb * xb[i];
            r.v[i] = from_float<T>(v);
        }
        if constexpr (kVec) {
            *reinterpret_cast<V *>(oo + s * D + lane * E) = r;
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) oo[s * D + lane * E + i] = r.v[i];
        }
        if (lane == 0) lo[s] = lse;
    }
}

template <int D, typename T>
int launch_t(const void *oa, const float *la, const void *ob, const float *lb, void *oo, float *lo, int64_t n,
             cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(BSP_ERR_CUDA, "no current CUDA device");
    const int64_t warps_needed = n;
    int64_t blocks = (warps_needed + 7) / 8;
    blocks = blocks < 1 ? 1 : blocks > (int64_t)sms * 8 ? (int64_t)sms * 8 : blocks;
    constexpr uintptr_t kVecBytes = sizeof(T) * (D / 32);
    const bool vec = (reinterpret_cast<uintptr_t>(oa) | reinterpret_cast<uintptr_t>(ob) |
                      reinterpret_cast<uintptr_t>(oo)) % kVecBytes == 0;
    auto kern = vec ? merge_state_kernel<D, T, true> : merge_state_kernel<D, T, false>;
    kern<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const T *>(oa), la, static_cast<const T *>(ob), lb,
                                               static_cast<T *>(oo), lo, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("merge_state launch: ") + cudaGetErrorString(e));
    return BSP_OK;
}

}  // namespace

int launch_merge_state(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b, void *o_out,
                       float *lse_out, int64_t n_rows, int32_t num_heads, int32_t head_dim, int32_t dtype,
                       cudaStream_t stream) {
    const int64_t n = n_rows * num_heads;
    if (n == 0) return BSP_OK;
    const bool bf = dtype == BSP_DTYPE_BF16;
    switch (head_dim) {
        case 32: return bf ? launch_t<32, __nv_bfloat16>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream)
                           : launch_t<32, float>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream);
        case 64: return bf ? launch_t<64, __nv_bfloat16>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream)
                           : launch_t<64, float>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream);
        case 128: return bf ? launch_t<128, __nv_bfloat16>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream)
                            : launch_t<128, float>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream);
        case 256: return bf ? launch_t<256, __nv_bfloat16>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream)
                            : launch_t<256, float>(o_a, lse_a, o_b, lse_b, o_out, lse_out, n, stream);
        default: return fail(BSP_ERR_UNSUPPORTED, "merge_state supports head_dim 32, 64, 128, 256");
    }
}

}  // namespace bsp
