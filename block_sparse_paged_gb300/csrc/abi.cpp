// C-ABI entry points of libbsp.so other than the planner: argument checks,
// launch of the run kernels, merge_state, error reporting.
#include <cstring>
#include <string>

#include "bsp_internal.h"

namespace bsp {

namespace {
thread_local std::string g_msg;
thread_local int g_code = BSP_OK;
}  // namespace

int fail(int code, const std::string &msg) {
    g_code = code;
    g_msg = msg;
    return code;
}

void clear_error() {
    g_code = BSP_OK;
    g_msg.clear();
}

int last_code() { return g_code == BSP_OK ? BSP_ERR_INVALID_ARG : g_code; }

int check_aligned16(const void *q, const void *k, const void *v, const void *o, const void *workspace) {
    const void *ptr[5] = {q, k, v, o, workspace};
    const char *name[5] = {"q", "k_pages", "v_pages", "o", "workspace"};
    for (int i = 0; i < 5; ++i)
        if (reinterpret_cast<uintptr_t>(ptr[i]) % 16 != 0)
            return fail(BSP_ERR_INVALID_ARG, std::string(name[i]) + " is not 16-byte aligned");
    return BSP_OK;
}

namespace {

int check_plan(const bsp_plan_info *plan, int mode, const void *workspace) {
    if (!plan || plan->valid != 1) return fail(BSP_ERR_INVALID_ARG, "plan is NULL or was not produced by bsp_plan");
    if (plan->problem.mode != mode)
        return fail(BSP_ERR_INVALID_ARG, mode == BSP_MODE_DECODE ? "plan was made for prefill, not decode"
                                                                 : "plan was made for decode, not prefill");
    if (!workspace) return fail(BSP_ERR_INVALID_ARG, "workspace is NULL");
    Layout l;
    if (!compute_layout(&plan->problem, &plan->capacity, &l)) return last_code();
    if (l.total != plan->workspace_bytes || l.off_partial_o != plan->off_partial_o)
        return fail(BSP_ERR_INVALID_ARG, "plan info is inconsistent with its problem and capacity");
    return BSP_OK;
}

}  // namespace
}  // namespace bsp

using namespace bsp;

extern "C" const char *bsp_last_error(void) { return g_msg.c_str(); }

extern "C" const char *bsp_version(void) { return "bsp 0.1 (sm_103a)"; }

extern "C" int bsp_default_num_ctas(int32_t mode, int32_t device, int32_t *num_ctas_out) {
    clear_error();
    if (!num_ctas_out) return fail(BSP_ERR_INVALID_ARG, "num_ctas_out is NULL");
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("device query: ") + cudaGetErrorString(e));
    if (mode == BSP_MODE_DECODE) *num_ctas_out = sms * decode_ctas_per_sm(128, BSP_DTYPE_BF16);
    else if (mode == BSP_MODE_PREFILL) *num_ctas_out = sms;
    else return fail(BSP_ERR_INVALID_ARG, "unknown mode");
    return BSP_OK;
}

extern "C" int bsp_decode_run(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *kv_indices, int64_t num_pages, float sm_scale, void *o, float *lse,
                              void *workspace, bsp_stream_t stream) {
    clear_error();
    int rc = check_plan(plan, BSP_MODE_DECODE, workspace);
    if (rc != BSP_OK) return rc;
    if (!q || !k_pages || !v_pages || !o) return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (num_pages < 0) return fail(BSP_ERR_INVALID_ARG, "num_pages must not be negative");
    if ((rc = check_aligned16(q, k_pages, v_pages, o, workspace)) != BSP_OK) return rc;
    // split outputs are merged inside the decode kernel (by the CTA that writes
    // an output's last partial state): one launch
    return launch_decode(plan, q, k_pages, v_pages, kv_indices, num_pages, sm_scale, o, lse, workspace, stream);
}

extern "C" int bsp_decode_run_fp8(const bsp_plan_info *plan, const void *q, const void *k_pages,
                                  const void *v_pages, const int32_t *kv_indices, int64_t num_pages, float sm_scale,
                                  float k_scale, float v_scale, void *o, float *lse, void *workspace,
                                  bsp_stream_t stream) {
    clear_error();
    int rc = check_plan(plan, BSP_MODE_DECODE, workspace);
    if (rc != BSP_OK) return rc;
    if (!q || !k_pages || !v_pages || !o) return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if ((rc = check_aligned16(q, k_pages, v_pages, o, workspace)) != BSP_OK) return rc;
    return launch_decode_fp8(plan, q, k_pages, v_pages, kv_indices, num_pages, sm_scale, k_scale, v_scale, o, lse,
                             workspace, stream);
}

extern "C" int bsp_prefill_run(const bsp_plan_info *plan, const void *q, const void *k_pages, const void *v_pages,
                               const int32_t *kv_indices, int64_t num_pages, float sm_scale, void *o, float *lse,
                               void *workspace, bsp_stream_t stream) {
    clear_error();
    int rc = check_plan(plan, BSP_MODE_PREFILL, workspace);
    if (rc != BSP_OK) return rc;
    if (!q || !k_pages || !v_pages || !o) return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (num_pages < 1) return fail(BSP_ERR_INVALID_ARG, "num_pages must be positive");
    if ((rc = check_aligned16(q, k_pages, v_pages, o, workspace)) != BSP_OK) return rc;
    rc = launch_prefill(plan, q, k_pages, v_pages, kv_indices, num_pages, sm_scale, o, lse, workspace, stream);
    if (rc != BSP_OK) return rc;
    return launch_reduce(plan, o, lse, workspace, stream);
}

extern "C" int bsp_run_attention(const bsp_plan_info *plan, const void *q, const void *k_pages,
                                 const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                                 float sm_scale, void *o, float *lse, void *workspace, bsp_stream_t stream) {
    clear_error();
    if (!plan) return fail(BSP_ERR_INVALID_ARG, "plan is NULL");
    const int mode = plan->problem.mode;
    int rc = check_plan(plan, mode, workspace);
    if (rc != BSP_OK) return rc;
    if (!q || !k_pages || !v_pages || !o) return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if ((rc = check_aligned16(q, k_pages, v_pages, o, workspace)) != BSP_OK) return rc;
    if (mode == BSP_MODE_DECODE) {
        if (num_pages < 0) return fail(BSP_ERR_INVALID_ARG, "num_pages must not be negative");
        return launch_decode(plan, q, k_pages, v_pages, kv_indices, num_pages, sm_scale, o, lse, workspace, stream);
    }
    if (num_pages < 1) return fail(BSP_ERR_INVALID_ARG, "num_pages must be positive");
    return launch_prefill(plan, q, k_pages, v_pages, kv_indices, num_pages, sm_scale, o, lse, workspace, stream);
}

extern "C" int bsp_run_merge_partials(const bsp_plan_info *plan, void *o, float *lse, void *workspace,
                                      bsp_stream_t stream) {
    clear_error();
    if (!plan) return fail(BSP_ERR_INVALID_ARG, "plan is NULL");
    int rc = check_plan(plan, plan->problem.mode, workspace);
    if (rc != BSP_OK) return rc;
    if (!o) return fail(BSP_ERR_INVALID_ARG, "o is NULL");
    return launch_reduce(plan, o, lse, workspace, stream);
}

extern "C" int bsp_check_bounded_wait(int64_t limit_cycles, int32_t *status, bsp_stream_t stream) {
    clear_error();
    if (!status) return fail(BSP_ERR_INVALID_ARG, "status is NULL");
    if (limit_cycles < 1 || limit_cycles > (int64_t{1} << 33))
        return fail(BSP_ERR_INVALID_ARG, "limit_cycles must be in [1, 2^33] (about 4 s)");
    return launch_wait_probe(limit_cycles, reinterpret_cast<int *>(status), stream);
}

extern "C" int bsp_merge_state(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b, void *o_out,
                               float *lse_out, int64_t n_rows, int32_t num_heads, int32_t head_dim, int32_t dtype,
                               bsp_stream_t stream) {
    clear_error();
    if (n_rows < 0 || num_heads < 1 || head_dim < 1) return fail(BSP_ERR_INVALID_ARG, "bad merge_state sizes");
    if (dtype != BSP_DTYPE_BF16 && dtype != BSP_DTYPE_F32) return fail(BSP_ERR_INVALID_ARG, "bad dtype");
    if (n_rows > 0 && (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out))
        return fail(BSP_ERR_INVALID_ARG, "a tensor pointer is NULL");
    return launch_merge_state(o_a, lse_a, o_b, lse_b, o_out, lse_out, n_rows, num_heads, head_dim, dtype, stream);
}

extern "C" int bsp_check_device_error(const bsp_plan_info *plan, void *workspace, bsp_stream_t stream,
                                      int32_t *word_out) {
    clear_error();
    if (!word_out) return fail(BSP_ERR_INVALID_ARG, "word_out is NULL");
    *word_out = 0;
    if (!plan || plan->valid != 1 || !workspace) return fail(BSP_ERR_INVALID_ARG, "plan or workspace missing");
    uint8_t *status = static_cast<uint8_t *>(workspace) + plan->off_status;
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, status, sizeof(word), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && word != 0) {
        e = cudaMemsetAsync(status, 0, sizeof(word), stream);
        // CTAs that gave up may have left partial counts in the reduction map's
        // arrival words; a later run of this plan would then fold too early
        if (e == cudaSuccess && plan->num_merges > 0)
            e = cudaMemset2DAsync(static_cast<uint8_t *>(workspace) + plan->off_merges +
                                      offsetof(bsp_merge_entry, arrived),
                                  sizeof(bsp_merge_entry), 0, sizeof(int32_t), (size_t)plan->num_merges, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    if (e != cudaSuccess) return fail(BSP_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
    *word_out = word;
    return BSP_OK;
}
