// tmap.cuh -- tensor-map (TMA descriptor) encoding for the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace spc {

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

// cuTensorMapEncodeTiled, looked up once through the runtime (no libcuda link).
inline EncodeFn tmap_encoder()
{
    static EncodeFn fn = []() -> EncodeFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

// 2-D row-major [rows, cols] tensor of `ebytes`-byte elements, boxes of
// box_cols x box_rows, with the given swizzle; false if it cannot be encoded.
inline bool tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int ebytes, const void* base,
                    uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                    CUtensorMapSwizzle swz)
{
    EncodeFn enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (uint64_t)ebytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace spc
