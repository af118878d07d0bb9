// Ragged causal prefill on the tensor cores (placeholder until the tcgen05
// kernel lands).
#include "bsp_internal.h"

namespace bsp {

int launch_prefill(const bsp_plan_info *, const void *, const void *, const void *, const int32_t *, int64_t,
                   float, void *, float *, void *, cudaStream_t) {
    return fail(BSP_ERR_UNSUPPORTED, "prefill kernel not built yet");
}

}  // namespace bsp
