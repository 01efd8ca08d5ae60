// Host-side tensor-map encoding (the driver's cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query; no link against libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace sgemm {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major fp32 matrix (rows x cols, leading dimension ld elements) as a 2-D
// tensor map with boxes of box_cols x box_rows, zero fill outside the matrix.
// swizzle_bytes: 0 (none), 64 or 128 (the box row must not be wider).
inline bool encode_fp32_2d(CUtensorMap* tm, const float* base, long long rows, long long cols,
                           long long ld, int box_cols, int box_rows, int swizzle_bytes) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
              : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                    : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace sgemm
