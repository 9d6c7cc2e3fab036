// rows.cu -- a row order of an indice map that groups rows by offset mask.
//
// A row's mask has bit k set when map[k, row] != -1.  Rows sorted by mask (a
// stable radix sort of (mask << 32 | row), so rows keep their order within a
// group) put rows that use the same offsets next to each other.  The tensor-
// core conv computes its 256-row tiles in this order, and a tile then runs only
// the offsets of its group: for the transposed map of a stride-2 k3 conv (the
// inverse conv's map) each of the eight parity classes of rows uses 1, 2, 4 or
// 8 of the 27 offsets, where a tile of consecutive rows mixes all of them.
#include "kernels.cuh"

namespace spc {

namespace {

constexpr int kBlock = 256;

__global__ void __launch_bounds__(kBlock)
k_row_mask_keys(const int32_t* __restrict__ map, int K, int64_t n, uint32_t* __restrict__ mask,
                unsigned long long* __restrict__ keys, unsigned long long* __restrict__ counter)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *counter = (unsigned long long)n;
    if (i >= n) return;
    uint32_t bits = 0;
    for (int k = 0; k < K; ++k)
        if (__ldg(map + (int64_t)k * n + i) >= 0) bits |= 1u << k;
    if (mask) mask[i] = bits;
    keys[i] = ((unsigned long long)bits << 32) | (unsigned long long)i;
}

// Keys from masks a build already wrote (no map read).
__global__ void __launch_bounds__(kBlock)
k_row_keys_from_mask(const uint32_t* __restrict__ mask, int K, int64_t n,
                     unsigned long long* __restrict__ keys, unsigned long long* __restrict__ counter)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *counter = (unsigned long long)n;
    if (i >= n) return;
    const uint32_t bits = __ldg(mask + i) & (K >= 32 ? 0xffffffffu : ((1u << K) - 1u));
    keys[i] = ((unsigned long long)bits << 32) | (unsigned long long)i;
}

__global__ void __launch_bounds__(kBlock)
k_perm_from_keys(const unsigned long long* __restrict__ keys, int64_t n, int32_t* __restrict__ perm)
{
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j < n) perm[j] = (int32_t)(keys[j] & 0xFFFFFFFFull);
}

struct RowWs {
    unsigned long long* counter;
    unsigned long long* keys_a;
    unsigned long long* keys_b;
    void* radix;
};

size_t carve(int64_t n, char* base, RowWs* w)
{
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off = align_up(off + bytes, 256);
        return p;
    };
    char* c = take(sizeof(unsigned long long));
    char* a = take(sizeof(unsigned long long) * (size_t)(n > 0 ? n : 1));
    char* b = take(sizeof(unsigned long long) * (size_t)(n > 0 ? n : 1));
    char* r = take(radix_ws_bytes(n));
    if (w) {
        w->counter = reinterpret_cast<unsigned long long*>(c);
        w->keys_a = reinterpret_cast<unsigned long long*>(a);
        w->keys_b = reinterpret_cast<unsigned long long*>(b);
        w->radix = r;
    }
    return off;
}

}  // namespace

size_t row_order_ws_bytes(int64_t n) { return carve(n, nullptr, nullptr); }

spc_status map_row_order(const int32_t* map, int32_t K, int64_t n, uint32_t* mask, int32_t* perm,
                         void* ws, size_t ws_bytes, cudaStream_t st)
{
    if (n == 0) return SPC_OK;
    if (!ws || ws_bytes < row_order_ws_bytes(n)) return SPC_ERR_WORKSPACE;
    RowWs w;
    carve(n, static_cast<char*>(ws), &w);
    const unsigned grid = (unsigned)ceil_div(n, (int64_t)kBlock);
    if (map)
        k_row_mask_keys<<<grid, kBlock, 0, st>>>(map, K, n, mask, w.keys_a, w.counter);
    else
        k_row_keys_from_mask<<<grid, kBlock, 0, st>>>(mask, K, n, w.keys_a, w.counter);
    SPC_LAUNCH_CHECK();
    const spc_status s = radix_sort_keys(w.keys_a, w.keys_b, w.counter, n, 32, 32 + K, w.radix, st);
    if (s != SPC_OK) return s;
    k_perm_from_keys<<<grid, kBlock, 0, st>>>(w.keys_a, n, perm);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace spc
