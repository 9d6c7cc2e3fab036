// maxpool.cu -- sparse max pooling on a strided indice map (spconv SparseMaxPool3d).
//
// Forward: out[o, c] = the largest x[i, c] over the pairs imap[k, o] = i (the
// occupied inputs of o's window only), and, when asked, arg[o, c] = the first
// offset k reaching it.  Backward: dx[i, c] = the sum of dy[o, c] over the
// pairs (k, o) of row i whose output picked k for channel c; read input-
// stationary through the transposed map, so every row of dx is written once,
// without atomics, in a fixed order.
//
// A thread owns one row and V consecutive channels (16 bytes when the row
// length allows vector loads); a warp covers whole rows, so each neighbour row
// is read as full 16-byte words.  Both kernels are bound by the gathers.
#include "kernels.cuh"

namespace spc {

namespace {

constexpr int kBlock = 256;
constexpr uint8_t kNoPair = 255;

template <typename T, int V>
struct Vec {
    T e[V];
};

template <typename T, int V>
__device__ __forceinline__ void load_vec(Vec<T, V>& v, const T* __restrict__ p)
{
    if constexpr (V * sizeof(T) == 16) {
        *reinterpret_cast<uint4*>(v.e) = __ldg(reinterpret_cast<const uint4*>(p));
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) v.e[j] = p[j];
    }
}

template <typename T, int V>
__global__ void __launch_bounds__(kBlock)
k_maxpool_fwd(const T* __restrict__ x, const int32_t* __restrict__ imap,
              const uint32_t* __restrict__ mask, int K, int64_t n_in, int64_t n_out, int c,
              T* __restrict__ y, uint8_t* __restrict__ arg)
{
    const int groups = c / V;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_out * groups) return;
    const int64_t o = t / groups;
    const int c0 = (int)(t % groups) * V;
    float best[V];
    uint8_t kbest[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        best[j] = 0.f;
        kbest[j] = kNoPair;
    }
    const uint32_t m = mask ? __ldg(mask + o) : 0u;
    for (int k = 0; k < K; ++k) {
        if (mask && !((m >> k) & 1u)) continue;
        const int32_t i = __ldg(imap + (int64_t)k * n_out + o);
        if (i < 0 || i >= n_in) continue;
        Vec<T, V> v;
        load_vec<T, V>(v, x + (int64_t)i * c + c0);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const float f = elem<T>::to_f32(v.e[j]);
            if (kbest[j] == kNoPair || f > best[j]) {  // the first offset wins ties
                best[j] = f;
                kbest[j] = (uint8_t)k;
            }
        }
    }
    Vec<T, V> out;
#pragma unroll
    for (int j = 0; j < V; ++j) out.e[j] = elem<T>::from_f32(best[j]);  // exact: a max of dt values
    T* dst = y + o * c + c0;
    if constexpr (V * sizeof(T) == 16) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(out.e);
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) dst[j] = out.e[j];
    }
    if (arg) {
#pragma unroll
        for (int j = 0; j < V; ++j) arg[o * c + c0 + j] = kbest[j];
    }
}

template <typename T, int V>
__global__ void __launch_bounds__(kBlock)
k_maxpool_dgrad(const T* __restrict__ dy, const int32_t* __restrict__ imap_t,
                const uint8_t* __restrict__ arg, int K, int64_t n_in, int64_t n_out, int c,
                T* __restrict__ dx)
{
    const int groups = c / V;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_in * groups) return;
    const int64_t i = t / groups;
    const int c0 = (int)(t % groups) * V;
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    for (int k = 0; k < K; ++k) {
        const int32_t o = __ldg(imap_t + (int64_t)k * n_in + i);
        if (o < 0 || o >= n_out) continue;
        Vec<T, V> g;
        load_vec<T, V>(g, dy + (int64_t)o * c + c0);
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (__ldg(arg + (int64_t)o * c + c0 + j) == (uint8_t)k) acc[j] += elem<T>::to_f32(g.e[j]);
    }
    Vec<T, V> out;
#pragma unroll
    for (int j = 0; j < V; ++j) out.e[j] = elem<T>::from_f32(acc[j]);
    T* dst = dx + i * c + c0;
    if constexpr (V * sizeof(T) == 16) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(out.e);
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) dst[j] = out.e[j];
    }
}

template <typename T>
spc_status launch_fwd(const void* x, const int32_t* imap, const uint32_t* mask, int K, int64_t n_in,
                      int64_t n_out, int c, void* y, uint8_t* arg, cudaStream_t st)
{
    constexpr int V16 = 16 / (int)sizeof(T);
    const bool vec = c % V16 == 0 && aligned16(x) && aligned16(y);
    const int64_t threads = n_out * (vec ? c / V16 : c);
    const unsigned grid = (unsigned)ceil_div(threads, (int64_t)kBlock);
    if (vec)
        k_maxpool_fwd<T, V16><<<grid, kBlock, 0, st>>>(static_cast<const T*>(x), imap, mask, K, n_in,
                                                       n_out, c, static_cast<T*>(y), arg);
    else
        k_maxpool_fwd<T, 1><<<grid, kBlock, 0, st>>>(static_cast<const T*>(x), imap, mask, K, n_in,
                                                     n_out, c, static_cast<T*>(y), arg);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

template <typename T>
spc_status launch_dgrad(const void* dy, const int32_t* imap_t, const uint8_t* arg, int K, int64_t n_in,
                        int64_t n_out, int c, void* dx, cudaStream_t st)
{
    constexpr int V16 = 16 / (int)sizeof(T);
    const bool vec = c % V16 == 0 && aligned16(dy) && aligned16(dx);
    const int64_t threads = n_in * (vec ? c / V16 : c);
    const unsigned grid = (unsigned)ceil_div(threads, (int64_t)kBlock);
    if (vec)
        k_maxpool_dgrad<T, V16><<<grid, kBlock, 0, st>>>(static_cast<const T*>(dy), imap_t, arg, K,
                                                         n_in, n_out, c, static_cast<T*>(dx));
    else
        k_maxpool_dgrad<T, 1><<<grid, kBlock, 0, st>>>(static_cast<const T*>(dy), imap_t, arg, K,
                                                       n_in, n_out, c, static_cast<T*>(dx));
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace

spc_status maxpool_fwd(const void* x, const int32_t* imap, const uint32_t* mask, int32_t K,
                       int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* y, uint8_t* arg,
                       cudaStream_t st)
{
    if (n_out == 0 || c == 0) return SPC_OK;
    switch (dt) {
    case SPC_F32: return launch_fwd<float>(x, imap, mask, K, n_in, n_out, c, y, arg, st);
    case SPC_F16: return launch_fwd<__half>(x, imap, mask, K, n_in, n_out, c, y, arg, st);
    case SPC_BF16: return launch_fwd<__nv_bfloat16>(x, imap, mask, K, n_in, n_out, c, y, arg, st);
    }
    return SPC_ERR_INVALID_ARG;
}

spc_status maxpool_dgrad(const void* dy, const int32_t* imap_t, const uint8_t* arg, int32_t K,
                         int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* dx,
                         cudaStream_t st)
{
    if (n_in == 0 || c == 0) return SPC_OK;
    switch (dt) {
    case SPC_F32: return launch_dgrad<float>(dy, imap_t, arg, K, n_in, n_out, c, dx, st);
    case SPC_F16: return launch_dgrad<__half>(dy, imap_t, arg, K, n_in, n_out, c, dx, st);
    case SPC_BF16: return launch_dgrad<__nv_bfloat16>(dy, imap_t, arg, K, n_in, n_out, c, dx, st);
    }
    return SPC_ERR_INVALID_ARG;
}

}  // namespace spc
