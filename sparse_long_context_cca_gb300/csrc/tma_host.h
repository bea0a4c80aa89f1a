// Host-side TMA descriptor encoding shared by the tensor-core kernels.
// cuTensorMapEncodeTiled is fetched through the runtime's driver entry point, so
// the library does not link against libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace cca {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encoder() {
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

// A bf16 tensor [heads, rows, 128] viewed as 3-D (128, rows, heads); box = 64 columns
// x 128 rows x 1 head with 128-byte swizzle.  Rows past `rows` read as zeros.
inline bool encode_3d_bf16_d128(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, uint64_t rows,
                                uint64_t heads) {
    const cuuint64_t dims[3] = {128, rows, heads};
    const cuuint64_t strides[2] = {128 * 2, rows * 128 * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An fp32 tensor [heads, rows, 128] viewed as 3-D (128, rows, heads); box = 32 columns
// (128 bytes) x 128 rows x 1 head with 128-byte swizzle, for tiled stores from shared
// memory.  Rows past `rows` are not written.
inline bool encode_3d_f32_d128(EncodeTiledFn enc, CUtensorMap *map, void *ptr, uint64_t rows, uint64_t heads) {
    const cuuint64_t dims[3] = {128, rows, heads};
    const cuuint64_t strides[2] = {128 * 4, rows * 128 * 4};
    const cuuint32_t box[3] = {32, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace cca
