// Host side of the TMA copies: 3-D bf16 tensor maps over [rows][heads][D]
// arrays (queries, outputs, paged K and V), encoded through the driver entry
// point that the runtime hands out (no link-time dependency on libcuda).
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "bsp_internal.h"

namespace bsp {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

}  // namespace

int make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t dim, uint64_t heads, uint64_t rows, uint32_t box_heads,
                   uint32_t box_rows) {
    return make_tmap(map, base, 2, dim, heads, rows, box_heads, box_rows);
}

int make_tmap(CUtensorMap *map, const void *base, int elem_bytes, uint64_t dim, uint64_t heads, uint64_t rows,
              uint32_t box_heads, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(BSP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return fail(BSP_ERR_INVALID_ARG, "tensor base not 16-byte aligned");
    cuuint64_t dims[3] = {(cuuint64_t)dim, heads, rows};
    cuuint64_t strides[2] = {(cuuint64_t)dim * elem_bytes, heads * dim * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), box_heads, box_rows};  // 128-byte rows
    cuuint32_t es[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(*map));
    const CUtensorMapDataType ty = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = enc(map, ty, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(BSP_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return BSP_OK;
}

}  // namespace bsp
