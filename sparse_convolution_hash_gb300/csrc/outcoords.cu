// outcoords.cu -- output coordinate set of a strided sparse conv.
//
// When a bitmap of the output grid fits in the space the sort below keeps for
// its keys (one bit per output cell against 16 bytes per candidate), each
// candidate sets its cell's bit with an atomic OR instead; per-block popcounts,
// one scan and a write of the set bits in order give the same sorted, unique
// set in five launches.  Otherwise:
//
// Every (input voxel, kernel offset) pair that lands exactly on an output cell
// (i + pad - k*dil divisible by the stride, quotient inside the output grid)
// names that cell.  The candidate cell keys ((b*Do + z)*Ho + y)*Wo + x are
// appended to a list, sorted by a least-significant-digit radix sort over the
// key's significant bits only (8-bit digits, stable scatter), and adjacent
// duplicates are dropped; the survivors, decoded, are the output rows in
// (b, z, y, x) order.  Everything runs on the stream with no host round trip;
// the candidate count stays on the device and blocks past it do nothing.
#include "kernels.cuh"

namespace spc {

namespace {

constexpr int kThreads = 256;
constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;  // elements per sort / unique block
constexpr int kRadix = 256;
constexpr int kScanThreads = 1024;

struct OutGeom {
    int32_t in_shape[3];
    int32_t out_shape[3];
    int32_t ksize[3];
    int32_t stride[3];
    int32_t pad[3];
    int32_t dil[3];
    int32_t batch;
    int32_t K;
};

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(kThreads)
k_candidates(const int4* __restrict__ coords, int64_t n, OutGeom g,
             unsigned long long* __restrict__ keys, unsigned long long* __restrict__ counter,
             int32_t* __restrict__ status)
{
    const int lane = threadIdx.x & 31;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < n;
         base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = base + threadIdx.x;
        bool valid = i < n;
        int4 c = make_int4(0, 0, 0, 0);
        if (valid) {
            c = coords[i];
            if (c.x < 0 || c.x >= g.batch || c.y < 0 || c.y >= g.in_shape[0] || c.z < 0 ||
                c.z >= g.in_shape[1] || c.w < 0 || c.w >= g.in_shape[2]) {
                set_status(status, SPC_ERR_COORD_RANGE);
                valid = false;
            }
        }
        const int p[3] = {c.y, c.z, c.w};
        for (int k = 0; k < g.K; ++k) {
            const int ka[3] = {k / (g.ksize[2] * g.ksize[1]), (k / g.ksize[2]) % g.ksize[1],
                               k % g.ksize[2]};
            bool ok = valid;
            int o[3];
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int t = p[a] + g.pad[a] - ka[a] * g.dil[a];
                o[a] = t >= 0 ? t / g.stride[a] : -1;
                ok = ok && t >= 0 && (t - o[a] * g.stride[a]) == 0 && o[a] < g.out_shape[a];
            }
            const uint32_t bal = __ballot_sync(FULL_MASK, ok);
            if (bal == 0) continue;
            const int leader = __ffs(bal) - 1;
            unsigned long long basepos = 0;
            if (lane == leader) basepos = atomicAdd(counter, (unsigned long long)__popc(bal));
            basepos = __shfl_sync(FULL_MASK, basepos, leader);
            if (ok) {
                const unsigned long long key =
                    (((unsigned long long)c.x * g.out_shape[0] + (unsigned)o[0]) * g.out_shape[1] +
                     (unsigned)o[1]) * g.out_shape[2] + (unsigned)o[2];
                keys[basepos + __popc(bal & lanemask_lt())] = key;
            }
        }
    }
}

// Bitmap path: every candidate cell of every input voxel sets its bit.  Small
// grids (SMEM) mark a block-private copy in shared memory and merge its
// nonzero words once; large grids OR straight into global memory, one atomic
// per distinct word per warp (lanes hitting the same word combine first).
constexpr int kSmemWords = 8192;  // 32 KB: output grids of up to 262,144 cells

template <bool SMEM>
__global__ void __launch_bounds__(kThreads)
k_bm_mark(const int4* __restrict__ coords, int64_t n, OutGeom g, uint32_t* __restrict__ bm,
          int64_t words, int32_t* __restrict__ status)
{
    __shared__ uint32_t s_bm[SMEM ? kSmemWords : 1];
    if (SMEM) {
        for (int64_t j = threadIdx.x; j < words; j += blockDim.x) s_bm[j] = 0u;
        __syncthreads();
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // every lane runs the same number of rounds, so the warp stays converged
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < n; base += stride) {
        const int64_t i = base + threadIdx.x;
        bool valid = i < n;
        int4 c = make_int4(0, 0, 0, 0);
        if (valid) {
            c = coords[i];
            if (c.x < 0 || c.x >= g.batch || c.y < 0 || c.y >= g.in_shape[0] || c.z < 0 ||
                c.z >= g.in_shape[1] || c.w < 0 || c.w >= g.in_shape[2]) {
                set_status(status, SPC_ERR_COORD_RANGE);
                valid = false;
            }
        }
        const int p[3] = {c.y, c.z, c.w};
        for (int k = 0; k < g.K; ++k) {
            const int ka[3] = {k / (g.ksize[2] * g.ksize[1]), (k / g.ksize[2]) % g.ksize[1],
                               k % g.ksize[2]};
            bool ok = valid;
            int o[3];
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                const int t = p[a] + g.pad[a] - ka[a] * g.dil[a];
                o[a] = t >= 0 ? t / g.stride[a] : -1;
                ok = ok && t >= 0 && (t - o[a] * g.stride[a]) == 0 && o[a] < g.out_shape[a];
            }
            const unsigned long long key =
                ok ? (((unsigned long long)c.x * g.out_shape[0] + (unsigned)o[0]) * g.out_shape[1] +
                      (unsigned)o[1]) * g.out_shape[2] + (unsigned)o[2]
                   : 0ull;
            const uint32_t bit = ok ? 1u << (key & 31) : 0u;
            if (SMEM) {
                if (ok) atomicOr(&s_bm[key >> 5], bit);
            } else {
                // lanes of the same word OR their bits; the lowest of them writes
                const unsigned long long word = ok ? key >> 5 : ~0ull;
                const uint32_t same = __match_any_sync(FULL_MASK, word);
                const uint32_t bits = __reduce_or_sync(same, bit);
                if (ok && (threadIdx.x & 31) == __ffs(same) - 1) atomicOr(&bm[word], bits);
            }
        }
    }
    if (SMEM) {
        __syncthreads();
        for (int64_t j = threadIdx.x; j < words; j += blockDim.x)
            if (s_bm[j]) atomicOr(&bm[j], s_bm[j]);
    }
}

// Set bits of each block's kThreads words (one word per thread: a word can
// hold 32 output cells, so the write below is spread over as many threads).
__global__ void __launch_bounds__(kThreads)
k_bm_count(const uint32_t* __restrict__ bm, int64_t words, uint32_t* __restrict__ blocksum)
{
    __shared__ uint32_t s_sum;
    if (threadIdx.x == 0) s_sum = 0;
    __syncthreads();
    const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    uint32_t c = idx < words ? __popc(bm[idx]) : 0u;
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(FULL_MASK, c, d);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_sum, c);
    __syncthreads();
    if (threadIdx.x == 0) blocksum[blockIdx.x] = s_sum;
}

// Decodes the set bits, in order, at their scanned positions (thread j of a
// block owns word j of the block's words, so the block scan keeps the order).
__global__ void __launch_bounds__(kThreads)
k_bm_write(const uint32_t* __restrict__ bm, int64_t words, const uint32_t* __restrict__ blockoff,
           const unsigned long long* __restrict__ total, OutGeom g, int4* __restrict__ out,
           int64_t cap, int64_t* __restrict__ n_out, int32_t* __restrict__ status)
{
    __shared__ uint32_t s_warp[kThreads / 32];
    const int64_t wi = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    uint32_t bits = wi < words ? bm[wi] : 0u;
    const uint32_t cnt = __popc(bits);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL_MASK, inc, d);
        if (lane >= d) inc += t;
    }
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    uint32_t wbase = 0;
    for (int i = 0; i < w; ++i) wbase += s_warp[i];
    int64_t pos = (int64_t)blockoff[blockIdx.x] + wbase + inc - cnt;
    const unsigned W = (unsigned)g.out_shape[2], H = (unsigned)g.out_shape[1], D = (unsigned)g.out_shape[0];
    while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < cap) {
            const unsigned long long key = (unsigned long long)wi * 32ull + (unsigned)b;
            int4 c;
            if (key <= 0xFFFFFFFFull) {  // 32-bit division when the cell index fits
                unsigned k32 = (unsigned)key;
                c.w = (int)(k32 % W);
                k32 /= W;
                c.z = (int)(k32 % H);
                k32 /= H;
                c.y = (int)(k32 % D);
                c.x = (int)(k32 / D);
            } else {
                unsigned long long k64 = key;
                c.w = (int)(k64 % W);
                k64 /= W;
                c.z = (int)(k64 % H);
                k64 /= H;
                c.y = (int)(k64 % D);
                c.x = (int)(k64 / D);
            }
            out[pos] = c;
        }
        ++pos;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t t = (int64_t)*total;
        *n_out = t;
        if (t > cap) set_status(status, SPC_ERR_CAPACITY);
    }
}

__global__ void __launch_bounds__(kThreads)
k_radix_hist(const unsigned long long* __restrict__ keys,
             const unsigned long long* __restrict__ counter, int shift,
             uint32_t* __restrict__ hist, int nblocks)
{
    __shared__ uint32_t s_h[kRadix];
    s_h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t n = (int64_t)*counter;
    const int64_t start = (int64_t)blockIdx.x * kTile;
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = start + (int64_t)j * kThreads + threadIdx.x;
        if (idx < n) atomicAdd(&s_h[(keys[idx] >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    hist[(size_t)threadIdx.x * nblocks + blockIdx.x] = s_h[threadIdx.x];
}

// Exclusive scan of len uint32 values in place, one block; the total goes to
// *total when total != NULL.
__global__ void __launch_bounds__(kScanThreads)
k_scan_exclusive(uint32_t* __restrict__ v, int64_t len, unsigned long long* __restrict__ total)
{
    __shared__ uint32_t s_warp[kScanThreads / 32];
    const int64_t per = (len + kScanThreads - 1) / kScanThreads;
    const int64_t lo = (int64_t)threadIdx.x * per;
    const int64_t hi = lo + per < len ? lo + per : len;
    uint32_t sum = 0;
    for (int64_t j = lo; j < hi; ++j) sum += v[j];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL_MASK, inc, d);
        if (lane >= d) inc += t;
    }
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    if (w == 0) {
        uint32_t x = s_warp[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t = __shfl_up_sync(FULL_MASK, x, d);
            if (lane >= d) x += t;
        }
        s_warp[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    uint32_t run = inc - sum + (w > 0 ? s_warp[w - 1] : 0u);
    for (int64_t j = lo; j < hi; ++j) {
        const uint32_t t = v[j];
        v[j] = run;
        run += t;
    }
    if (total && threadIdx.x == kScanThreads - 1) *total = run;
}

// Stable scatter of one 8-bit digit.  Each tile is walked in order, 256
// elements at a time; an element's position is its digit's running base for
// this block + the count of equal digits in lower warps + in lower lanes.
__global__ void __launch_bounds__(kThreads)
k_radix_scatter(const unsigned long long* __restrict__ in, unsigned long long* __restrict__ out,
                const unsigned long long* __restrict__ counter, int shift,
                const uint32_t* __restrict__ hist, int nblocks)
{
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t s_base[kRadix];
    __shared__ uint32_t s_wcnt[kWarps][kRadix];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    (void)lane;
    const int64_t n = (int64_t)*counter;
    const int64_t start = (int64_t)blockIdx.x * kTile;
    if (start >= n) return;  // block-uniform
    s_base[threadIdx.x] = hist[(size_t)threadIdx.x * nblocks + blockIdx.x];
    const uint32_t lt = lanemask_lt();
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = start + (int64_t)j * kThreads + threadIdx.x;
        const bool valid = idx < n;
        const unsigned long long key = valid ? in[idx] : 0ull;
        const uint32_t d = valid ? (uint32_t)((key >> shift) & 0xFF) : (uint32_t)kRadix;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s_wcnt[w][threadIdx.x] = 0;
        __syncthreads();
        const uint32_t peers = __match_any_sync(FULL_MASK, d);
        const uint32_t rank = __popc(peers & lt);
        if (valid && rank == 0) s_wcnt[warp][d] = __popc(peers);
        __syncthreads();
        {
            uint32_t run = s_base[threadIdx.x];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t c = s_wcnt[w][threadIdx.x];
                s_wcnt[w][threadIdx.x] = run;
                run += c;
            }
            s_base[threadIdx.x] = run;
        }
        __syncthreads();
        if (valid) out[s_wcnt[warp][d] + rank] = key;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads)
k_unique_count(const unsigned long long* __restrict__ keys,
               const unsigned long long* __restrict__ counter, uint32_t* __restrict__ blocksum)
{
    __shared__ uint32_t s_sum;
    if (threadIdx.x == 0) s_sum = 0;
    __syncthreads();
    const int64_t n = (int64_t)*counter;
    const int64_t start = (int64_t)blockIdx.x * kTile;
    uint32_t c = 0;
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = start + (int64_t)j * kThreads + threadIdx.x;
        if (idx < n) c += (idx == 0 || keys[idx] != keys[idx - 1]) ? 1u : 0u;
    }
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(FULL_MASK, c, d);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_sum, c);
    __syncthreads();
    if (threadIdx.x == 0) blocksum[blockIdx.x] = s_sum;
}

// Writes the unique keys of each tile, decoded, at the tile's scanned offset.
// Each thread owns kItems consecutive elements so the block scan keeps order.
__global__ void __launch_bounds__(kThreads)
k_unique_write(const unsigned long long* __restrict__ keys,
               const unsigned long long* __restrict__ counter,
               const uint32_t* __restrict__ blockoff, const unsigned long long* __restrict__ total,
               OutGeom g, int4* __restrict__ out, int64_t cap, int64_t* __restrict__ n_out,
               int32_t* __restrict__ status)
{
    __shared__ uint32_t s_warp[kThreads / 32];
    const int64_t n = (int64_t)*counter;
    const int64_t start = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
    uint32_t flags = 0, cnt = 0;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = start + j;
        const bool f = idx < n && (idx == 0 || keys[idx] != keys[idx - 1]);
        flags |= (f ? 1u : 0u) << j;
        cnt += f ? 1u : 0u;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL_MASK, inc, d);
        if (lane >= d) inc += t;
    }
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    uint32_t wbase = 0;
    for (int i = 0; i < w; ++i) wbase += s_warp[i];
    int64_t pos = (int64_t)blockoff[blockIdx.x] + wbase + inc - cnt;
    for (int j = 0; j < kItems; ++j) {
        if (!((flags >> j) & 1u)) continue;
        if (pos < cap) {
            unsigned long long key = keys[start + j];
            int4 c;
            c.w = (int)(key % (unsigned)g.out_shape[2]);
            key /= (unsigned)g.out_shape[2];
            c.z = (int)(key % (unsigned)g.out_shape[1]);
            key /= (unsigned)g.out_shape[1];
            c.y = (int)(key % (unsigned)g.out_shape[0]);
            c.x = (int)(key / (unsigned)g.out_shape[0]);
            out[pos] = c;
        }
        ++pos;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t t = (int64_t)*total;
        *n_out = t;
        if (t > cap) set_status(status, SPC_ERR_CAPACITY);
    }
}

struct OutWs {
    unsigned long long* counter;  // [0] candidates, [1] unique total
    unsigned long long* keys_a;
    unsigned long long* keys_b;
    uint32_t* hist;
    uint32_t* blocksum;
};

int64_t cand_max(int64_t n_in, int32_t K) { return n_in * (int64_t)K; }

size_t carve(int64_t n_in, int32_t K, char* base, OutWs* w)
{
    const int64_t ncand = cand_max(n_in, K);
    const int64_t nblocks = ceil_div(ncand > 0 ? ncand : 1, kTile);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off = align_up(off + bytes, 256);
        return p;
    };
    char* c = take(2 * sizeof(unsigned long long));
    char* ka = take(sizeof(unsigned long long) * (size_t)(ncand > 0 ? ncand : 1));
    char* kb = take(sizeof(unsigned long long) * (size_t)(ncand > 0 ? ncand : 1));
    char* h = take(sizeof(uint32_t) * (size_t)kRadix * (size_t)nblocks);
    char* bs = take(sizeof(uint32_t) * (size_t)(nblocks + 1));
    if (w) {
        w->counter = reinterpret_cast<unsigned long long*>(c);
        w->keys_a = reinterpret_cast<unsigned long long*>(ka);
        w->keys_b = reinterpret_cast<unsigned long long*>(kb);
        w->hist = reinterpret_cast<uint32_t*>(h);
        w->blocksum = reinterpret_cast<uint32_t*>(bs);
    }
    return off;
}

}  // namespace

size_t outcoords_ws_bytes(int64_t n_in, int32_t K) { return carve(n_in, K, nullptr, nullptr); }

size_t radix_ws_bytes(int64_t n)
{
    const int64_t nblocks = ceil_div(n > 0 ? n : 1, (int64_t)kTile);
    return align_up(sizeof(uint32_t) * (size_t)kRadix * (size_t)nblocks, 256);
}

spc_status radix_sort_keys(unsigned long long* a, unsigned long long* b, const unsigned long long* counter,
                           int64_t n, int lo_bit, int hi_bit, void* ws, cudaStream_t st)
{
    if (n <= 1 || hi_bit <= lo_bit) return SPC_OK;
    const int nblocks = (int)ceil_div(n, (int64_t)kTile);
    uint32_t* hist = static_cast<uint32_t*>(ws);
    unsigned long long* src = a;
    unsigned long long* dst = b;
    for (int shift = lo_bit; shift < hi_bit; shift += 8) {
        k_radix_hist<<<nblocks, kThreads, 0, st>>>(src, counter, shift, hist, nblocks);
        SPC_LAUNCH_CHECK();
        k_scan_exclusive<<<1, kScanThreads, 0, st>>>(hist, (int64_t)kRadix * nblocks, nullptr);
        SPC_LAUNCH_CHECK();
        k_radix_scatter<<<nblocks, kThreads, 0, st>>>(src, dst, counter, shift, hist, nblocks);
        SPC_LAUNCH_CHECK();
        std::swap(src, dst);
    }
    if (src != a)
        SPC_CUDA_TRY(cudaMemcpyAsync(a, src, sizeof(unsigned long long) * (size_t)n,
                                     cudaMemcpyDeviceToDevice, st));
    return SPC_OK;
}

spc_status strided_out_coords(const int32_t* coords, int64_t n_in, const ProbeGeom& pg,
                              const int32_t out_shape[3], int32_t* out_coords, int64_t cap,
                              int64_t* n_out, int32_t* status, void* ws, size_t ws_bytes,
                              cudaStream_t st)
{
    if (!ws || ws_bytes < outcoords_ws_bytes(n_in, pg.K)) return SPC_ERR_WORKSPACE;
    OutWs w;
    carve(n_in, pg.K, static_cast<char*>(ws), &w);
    OutGeom g;
    for (int a = 0; a < 3; ++a) {
        g.in_shape[a] = pg.in_shape[a];
        g.out_shape[a] = out_shape[a];
        g.ksize[a] = pg.ksize[a];
        g.stride[a] = pg.stride[a];
        g.pad[a] = pg.pad[a];
        g.dil[a] = pg.dil[a];
    }
    g.batch = pg.batch;
    g.K = pg.K;
    SPC_CUDA_TRY(cudaMemsetAsync(w.counter, 0, 2 * sizeof(unsigned long long), st));
    const int64_t total_cells = (int64_t)pg.batch * out_shape[0] * out_shape[1] * out_shape[2];
    if (n_in == 0 || total_cells == 0) {
        SPC_CUDA_TRY(cudaMemsetAsync(n_out, 0, sizeof(int64_t), st));
        if (n_in > 0) {
            // still validate the inputs: no candidate can land anywhere
            const int grid = (int)std::min<int64_t>(ceil_div(n_in, kThreads), 8 * sm_count());
            OutGeom g0 = g;
            g0.K = 0;
            k_candidates<<<grid, kThreads, 0, st>>>(reinterpret_cast<const int4*>(coords), n_in,
                                                    g0, w.keys_a, w.counter, status);
            SPC_LAUNCH_CHECK();
        }
        return SPC_OK;
    }
    const int64_t ncand = cand_max(n_in, pg.K);
    const int64_t words = ceil_div(total_cells, (int64_t)32);
    if (words <= 2 * ncand) {
        // the bitmap takes the first key buffer, its block sums the second
        uint32_t* bm = reinterpret_cast<uint32_t*>(w.keys_a);
        uint32_t* bsum = reinterpret_cast<uint32_t*>(w.keys_b);
        const int nb = (int)ceil_div(words, (int64_t)kThreads);
        SPC_CUDA_TRY(cudaMemsetAsync(bm, 0, sizeof(uint32_t) * (size_t)words, st));
        const int grid = (int)std::min<int64_t>(ceil_div(n_in, kThreads), 8 * sm_count());
        if (words <= kSmemWords)
            k_bm_mark<true><<<grid, kThreads, 0, st>>>(reinterpret_cast<const int4*>(coords), n_in,
                                                       g, bm, words, status);
        else
            k_bm_mark<false><<<grid, kThreads, 0, st>>>(reinterpret_cast<const int4*>(coords), n_in,
                                                        g, bm, words, status);
        SPC_LAUNCH_CHECK();
        k_bm_count<<<nb, kThreads, 0, st>>>(bm, words, bsum);
        SPC_LAUNCH_CHECK();
        k_scan_exclusive<<<1, kScanThreads, 0, st>>>(bsum, nb, w.counter + 1);
        SPC_LAUNCH_CHECK();
        k_bm_write<<<nb, kThreads, 0, st>>>(bm, words, bsum, w.counter + 1, g,
                                            reinterpret_cast<int4*>(out_coords), cap, n_out,
                                            status);
        SPC_LAUNCH_CHECK();
        return SPC_OK;
    }
    const int nblocks = (int)ceil_div(ncand, kTile);
    {
        const int grid = (int)std::min<int64_t>(ceil_div(n_in, kThreads), 8 * sm_count());
        k_candidates<<<grid, kThreads, 0, st>>>(reinterpret_cast<const int4*>(coords), n_in, g,
                                                w.keys_a, w.counter, status);
        SPC_LAUNCH_CHECK();
    }
    const int bits = ceil_log2((uint64_t)total_cells);
    const int passes = (bits + 7) / 8;
    unsigned long long* src = w.keys_a;
    unsigned long long* dst = w.keys_b;
    for (int p = 0; p < passes; ++p) {
        k_radix_hist<<<nblocks, kThreads, 0, st>>>(src, w.counter, 8 * p, w.hist, nblocks);
        SPC_LAUNCH_CHECK();
        k_scan_exclusive<<<1, kScanThreads, 0, st>>>(w.hist, (int64_t)kRadix * nblocks, nullptr);
        SPC_LAUNCH_CHECK();
        k_radix_scatter<<<nblocks, kThreads, 0, st>>>(src, dst, w.counter, 8 * p, w.hist, nblocks);
        SPC_LAUNCH_CHECK();
        std::swap(src, dst);
    }
    k_unique_count<<<nblocks, kThreads, 0, st>>>(src, w.counter, w.blocksum);
    SPC_LAUNCH_CHECK();
    k_scan_exclusive<<<1, kScanThreads, 0, st>>>(w.blocksum, nblocks, w.counter + 1);
    SPC_LAUNCH_CHECK();
    k_unique_write<<<nblocks, kThreads, 0, st>>>(src, w.counter, w.blocksum, w.counter + 1, g,
                                                 reinterpret_cast<int4*>(out_coords), cap, n_out,
                                                 status);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace spc
