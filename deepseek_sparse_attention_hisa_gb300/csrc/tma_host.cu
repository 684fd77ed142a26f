// Host-side TMA tensor-map encoding. The encoder is a driver entry point fetched at run
// time, so libhisa links only the CUDA runtime statically and needs nothing but the
// driver when it loads.
#include <cudaTypedefs.h>

#include "hisa_internal.cuh"

namespace hisa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

}  // namespace

namespace {

bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, uint32_t esize, const void *base,
               uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encoder();
    if (!fn || rows == 0 || cols == 0) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};      // bytes between rows
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_bf16_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_cols, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_cols, box_rows);
}

bool encode_f32_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, box_cols, box_rows);
}

}  // namespace hisa
