// common.cuh -- shared device and host helpers of libspc (CUDA path only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "spc.h"

namespace spc {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Sticky error word: the first nonzero code written wins.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code)
{
    if (status) atomicCAS(status, (int32_t)SPC_OK, code);
}

// ---------------------------------------------------------------- element types
template <typename T> struct elem;
template <> struct elem<float> {
    static __device__ __forceinline__ float to_f32(float v) { return v; }
    static __device__ __forceinline__ float from_f32(float v) { return v; }
};
template <> struct elem<__half> {
    static __device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f32(float v) { return __float2half_rn(v); }
};
template <> struct elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// ------------------------------------------------------------- host utilities
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int ceil_log2(uint64_t v)
{
    int b = 0;
    while (b < 64 && (1ull << b) < v) ++b;
    return b;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessors of the current device (cached per device).
inline int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 1;
    }
    return cached[dev];
}

#define SPC_CUDA_TRY(expr)                                       \
    do {                                                         \
        cudaError_t _e = (expr);                                 \
        if (_e != cudaSuccess) return SPC_ERR_CUDA;              \
    } while (0)

#define SPC_LAUNCH_CHECK() SPC_CUDA_TRY(cudaGetLastError())

}  // namespace spc
