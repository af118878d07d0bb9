// Internal declarations shared by the translation units of libbsp.so:
// the workspace layout, the device-side plan header and error reporting.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/bsp.h"

namespace bsp {

constexpr int kPrefillTileRows = 256;   // packed query rows per prefill tile (two 128-row MMA subtiles)
constexpr int kMaxDecodeGroup = 16;     // decode tile: M = 16 rows of the MMA
constexpr uint64_t kAlign = 256;

// First 64 bytes of the workspace: what a kernel needs from the current plan.
struct DevHeader {
    int32_t num_items;
    int32_t num_merges;
    int32_t num_partials;
    int32_t tile_rows;
    int32_t group;
    int32_t num_ctas;
    int32_t chunk_len;
    int32_t reserved[9];
};
static_assert(sizeof(DevHeader) == 64, "DevHeader is 64 bytes");
static_assert(sizeof(bsp_work_item) == 64, "bsp_work_item is 64 bytes");
static_assert(sizeof(bsp_merge_entry) == 32, "bsp_merge_entry is 32 bytes");

// Offsets and capacities of the workspace sections; fixed by (problem, capacity).
struct Layout {
    int tile_rows = 0, group = 0;
    int64_t cap_tiles = 0;
    int64_t cap_items = 0, cap_merges = 0, cap_partials = 0;
    uint64_t off_header = 0, off_queue_indptr = 0, off_items = 0, off_merges = 0;
    uint64_t metadata_end = 0;  // staging buffer size
    uint64_t off_status = 0, off_partial_lse = 0, off_partial_o = 0;
    uint64_t off_gather = 0, gather_pool_bytes = 0;  // K copy region, then V (prefill, optional)
    uint64_t total = 0;
};

// Validates the static problem; returns false and sets the error message.
bool check_problem(const bsp_problem *p);
bool compute_layout(const bsp_problem *p, const bsp_capacity *c, Layout *out);

// Thread-local error message; returns `code` for convenient `return fail(...)`.
int fail(int code, const std::string &msg);
void clear_error();
// Code of the last fail() on this thread (BSP_ERR_INVALID_ARG if none).
int last_code();

inline uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// The run kernels move q, K / V rows, o and the workspace's partial states in
// 16-byte units: BSP_OK, or BSP_ERR_INVALID_ARG naming the first pointer that
// is not 16-byte aligned.
int check_aligned16(const void *q, const void *k, const void *v, const void *o, const void *workspace);

// 3-D bf16 TMA map over a [rows][heads][dim] array (dim a multiple of 64):
// boxes of 64 elements x box_heads x box_rows, 128-byte swizzle. BSP_OK or
// BSP_ERR_* (unaligned base, encoder unavailable or rejecting the shape).
int make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t dim, uint64_t heads, uint64_t rows, uint32_t box_heads,
                   uint32_t box_rows);
// The same for 1- or 2-byte elements: boxes of 128 / elem_bytes elements (one
// 128-byte swizzle row) x box_heads x box_rows.
int make_tmap(CUtensorMap *map, const void *base, int elem_bytes, uint64_t dim, uint64_t heads, uint64_t rows,
              uint32_t box_heads, uint32_t box_rows);

// Launchers (defined in the .cu files). They return BSP_OK or BSP_ERR_*.
int launch_decode(const bsp_plan_info *plan, const void *q, const void *k_pages,
                  const void *v_pages, const int32_t *kv_indices, int64_t num_pages, float sm_scale,
                  void *o, float *lse, void *workspace, cudaStream_t stream);
// Decode over e4m3 K/V pools with per-tensor scales (bf16 q and o).
int launch_decode_fp8(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *kv_indices, int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                      void *o, float *lse, void *workspace, cudaStream_t stream);
int launch_prefill(const bsp_plan_info *plan, const void *q, const void *k_pages,
                   const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                   float sm_scale, void *o, float *lse, void *workspace, cudaStream_t stream);
// Copy the page table's first n_pages pages of K and V, in table order, into
// the plan's gather region (prefill with a region); ids outside [0, num_pages)
// give zero pages and set the workspace status word.
int launch_gather_pages(const bsp_plan_info *plan, const void *k_pages, const void *v_pages,
                        const int32_t *kv_indices, int64_t num_pages, void *workspace, cudaStream_t stream);
int launch_wait_probe(long long limit_cycles, int *status, cudaStream_t stream);
int launch_reduce(const bsp_plan_info *plan, void *o, float *lse, void *workspace,
                  cudaStream_t stream);
int launch_merge_state(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b,
                       void *o_out, float *lse_out, int64_t n_rows, int32_t num_heads,
                       int32_t head_dim, int32_t dtype, cudaStream_t stream);
int decode_ctas_per_sm(int head_dim, int dtype);

}  // namespace bsp
