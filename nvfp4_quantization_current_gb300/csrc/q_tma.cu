// Host side of the tile engine: TMA tensor maps, encoded through the driver
// entry point that the runtime hands out (no link-time dependency on the
// driver library, so libq.so also loads on machines without a GPU).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

cudaError_t make_tile_map(void *map, const void *x, int dt, int64_t M, int64_t K, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    // A byte matrix is described as 16-bit elements (K/2 per row, K even):
    // a box edge may not exceed 256 elements, and 512 bytes of U8 would.
    const int es = dt == F32 ? 4 : 2;
    const CUtensorMapDataType ty = dt == BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : (dt == F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16);
    cuuint64_t dims[2] = {(cuuint64_t)(dt == U8 ? K / 2 : K), (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(dt == U8 ? K : K * es)};
    cuuint32_t box[2] = {(cuuint32_t)(512 / es), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(static_cast<CUtensorMap *>(map), ty,
                    2, const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_store_map_u8(void *map, void *base, int64_t row_bytes, int64_t rows, int box_bytes, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace qk
