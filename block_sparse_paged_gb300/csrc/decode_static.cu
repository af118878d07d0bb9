// Decode run for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc on the path where they run attention:
// a serving engine whose KV-cache manager reserved nearly all of HBM up front
// for its own pool and forbids further allocation while it serves requests,
// or a plugin that its host hands only the input and output tensors, with no
// allocator to draw scratch from. Such a caller can still plan on the host
// and pass its inputs and outputs; this entry point then keeps the run's
// scratch (the plan metadata and the partial states of split outputs) in a
// fixed array in device memory that the library itself declares.
//
// The array is a file-scope __device__ variable of BSP_STATIC_WORKSPACE_BYTES:
// every GPU that loads the library holds it until the process exits. Its
// device address is looked up once per device with cudaGetSymbolAddress
// (host code must not use the variable's name as a device pointer).
#include <mutex>

#include "bsp_internal.h"

namespace bsp {
namespace {

static __device__ __align__(256) uint8_t g_static_workspace[BSP_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_static_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_workspace on the current device; the lookup runs
// once per device, with that device current.
int static_workspace_ptr(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(BSP_ERR_UNSUPPORTED, "device index beyond 63");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess || !p)
            return fail(BSP_ERR_CUDA, std::string("cudaGetSymbolAddress(static workspace): ") +
                                          (e != cudaSuccess ? cudaGetErrorString(e) : "null address"));
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return BSP_OK;
}

}  // namespace
}  // namespace bsp

using namespace bsp;

extern "C" int bsp_decode_run_static(const bsp_plan_info *plan, const void *host_staging, const void *q,
                                     const void *k_pages, const void *v_pages, const int32_t *kv_indices,
                                     float sm_scale, void *o, float *lse, bsp_stream_t stream) {
    clear_error();
    if (!plan || (plan->valid != 1 && plan->valid != 2))
        return fail(BSP_ERR_INVALID_ARG, "plan is NULL or was not produced by bsp_plan");
    if (plan->problem.mode != BSP_MODE_DECODE) return fail(BSP_ERR_INVALID_ARG, "plan was made for prefill, not decode");
    if (!host_staging) return fail(BSP_ERR_INVALID_ARG, "host_staging (the plan's staging image) is NULL");
    if (!q || !k_pages || !v_pages || !o) return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (check_aligned16(q, k_pages, v_pages, o, nullptr) != BSP_OK) return last_code();
    Layout l;
    if (!compute_layout(&plan->problem, &plan->capacity, &l)) return last_code();
    if (l.total != plan->workspace_bytes || l.off_partial_o != plan->off_partial_o)
        return fail(BSP_ERR_INVALID_ARG, "plan info is inconsistent with its problem and capacity");
    // The plan's counts and offsets decide where the copies below write into
    // the shared array: accept only those of the layout its bounds define.
    if (plan->off_header != l.off_header || plan->off_queue_indptr != l.off_queue_indptr || plan->off_items != l.off_items ||
        plan->off_merges != l.off_merges || plan->off_status != l.off_status ||
        plan->off_partial_lse != l.off_partial_lse || plan->num_items < 0 || plan->num_items > l.cap_items ||
        plan->num_merges < 0 || plan->num_merges > l.cap_merges)
        return fail(BSP_ERR_INVALID_ARG, "plan info is inconsistent with its problem and capacity");
    if (plan->workspace_bytes > BSP_STATIC_WORKSPACE_BYTES)
        return fail(BSP_ERR_CAPACITY, "the plan's workspace (bsp_workspace_size) exceeds the static workspace "
                                      "BSP_STATIC_WORKSPACE_BYTES (8 MiB); lower capacity.num_ctas or max_batch, "
                                      "or use bsp_decode_run with a workspace of your own");
    void *ws = nullptr;
    int rc = static_workspace_ptr(&ws);
    if (rc != BSP_OK) return rc;

    // The array keeps whatever the previous call left: copy this plan's
    // metadata over it and clear the status word. Partial slots need no
    // clearing: each is written by its work item before the merge reads it.
    uint8_t *dst = static_cast<uint8_t *>(ws);
    const uint8_t *src = static_cast<const uint8_t *>(host_staging);
    cudaError_t e = cudaMemcpyAsync(dst, src, plan->off_items, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && plan->num_items > 0)
        e = cudaMemcpyAsync(dst + plan->off_items, src + plan->off_items,
                            sizeof(bsp_work_item) * (size_t)plan->num_items, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && plan->num_merges > 0)
        e = cudaMemcpyAsync(dst + plan->off_merges, src + plan->off_merges,
                            sizeof(bsp_merge_entry) * (size_t)plan->num_merges, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dst + plan->off_status, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("static plan copy: ") + cudaGetErrorString(e));
    // no pool size here, so no tensor maps: pages are gathered with cp.async
    // split outputs are merged inside the decode kernel
    return launch_decode(plan, q, k_pages, v_pages, kv_indices, 0, sm_scale, o, lse, ws, stream);
}
