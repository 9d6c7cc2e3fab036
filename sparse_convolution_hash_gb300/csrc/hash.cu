// hash.cu -- GPU open-addressing hash table over (b, z, y, x) cell keys and the
// indice-map probe kernel built on it.
//
// Keys: the mixed-radix cell index ((b*D + z)*H + y)*W + x over the grid (the
// int64 key of lato_mlx sparse/conv.py "build_indice_map", here bounded by an
// explicit range check instead of a pad shift).  A slot packs the key above the
// row index, so one 8-byte read both matches and resolves a probe.
//
// Buckets are 32 bytes (four slots, one L2 sector) and each lane reads a whole
// bucket per step with two 16-byte loads, so one read resolves nearly every
// lookup at load factor <= 1/2.  A warp works on 32 consecutive rows together:
// their coordinates arrive in one coalesced read, their map entries leave as
// 128-byte rows of imap, and the per-offset pair counts are one ballot per
// offset.  Inserts claim the first empty slot with a 64-bit CAS.  Every probe
// loop is bounded; exceeding the bound sets SPC_ERR_TABLE_FULL.
#include <algorithm>

#include "kernels.cuh"

namespace spc {

namespace {

constexpr unsigned long long EMPTY = ~0ull;
constexpr int kBlock = 256;

__device__ __forceinline__ uint32_t bucket_of(unsigned long long key, int log2b)
{
    const unsigned long long h = key * 0x9E3779B97F4A7C15ull;
    return log2b == 0 ? 0u : (uint32_t)(h >> (64 - log2b));
}

// Slot of the bucket an insert tries first (bits below the bucket index).
__device__ __forceinline__ int home_slot(unsigned long long key)
{
    return (int)(((key * 0x9E3779B97F4A7C15ull) >> 30) & 3u);
}

__device__ __forceinline__ unsigned long long cell_key(int b, int z, int y, int x, int D, int H,
                                                       int W)
{
    return (((unsigned long long)b * D + (unsigned)z) * H + (unsigned)y) * W + (unsigned)x;
}

// Fills every region of the list with its 32-bit pattern: the empty table, the
// zeroed pair counts and mask, and the map rows that start at -1.  One launch
// instead of a memset per buffer.  The 16-byte-aligned bodies of the regions
// form one index space that the grid strides over; the first threads also
// write each region's unaligned head and tail words.
__global__ void __launch_bounds__(kBlock) k_build_init(FillList L, int n)
{
    int64_t start[6];  // first 16-byte word of each region's body in the joint index space
    int64_t head[5];
    start[0] = 0;
    for (int i = 0; i < 5; ++i) {
        const FillRegion& f = L.r[i];
        const int64_t nn = i < n ? f.n : 0;
        head[i] = nn > 0 ? std::min<int64_t>(nn, (int64_t)((16 - (reinterpret_cast<uintptr_t>(f.p) & 15)) & 15) / 4) : 0;
        start[i + 1] = start[i] + (nn - head[i]) / 4;
    }
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t0 < 6 * 5) {  // heads (words 0..2) and tails (3..5) of region t0 / 6
        const int i = (int)(t0 / 6), w = (int)(t0 % 6);
        if (i < n && L.r[i].n > 0) {
            const FillRegion& f = L.r[i];
            const int64_t body_end = head[i] + (start[i + 1] - start[i]) * 4;
            const int64_t at = w < 3 ? w : body_end + (w - 3);
            if ((w < 3 && at < head[i]) || (w >= 3 && at < f.n)) f.p[at] = f.v;
        }
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int i = 0;
    for (int64_t j = t0; j < start[5]; j += stride) {
        while (j >= start[i + 1]) ++i;
        const FillRegion& f = L.r[i];
        reinterpret_cast<uint4*>(f.p + head[i])[j - start[i]] = make_uint4(f.v, f.v, f.v, f.v);
    }
}

// Reads one 32-byte bucket (four slots) with two 16-byte loads.
template <bool COHERENT>
__device__ __forceinline__ void load_bucket(const unsigned long long* slots, uint32_t bucket,
                                            unsigned long long v[4])
{
    const ulonglong2* b = reinterpret_cast<const ulonglong2*>(slots + (size_t)bucket * 4);
    ulonglong2 a, c;
    if (COHERENT) {
        a = __ldcg(b);
        c = __ldcg(b + 1);
    } else {
        a = __ldg(b);
        c = __ldg(b + 1);
    }
    v[0] = a.x;
    v[1] = a.y;
    v[2] = c.x;
    v[3] = c.y;
}

// One key per thread.  The thread reads its key's whole bucket at once; a slot
// holding the same key means a duplicate row, else it claims the first empty
// slot with a 64-bit CAS (re-reading the bucket if another thread won it), else
// it moves to the next bucket.  Bounded by 5 visits per bucket of the table.
__global__ void __launch_bounds__(kBlock)
k_hash_insert(const int4* __restrict__ coords, int64_t n, int32_t batch, int D, int H, int W,
              unsigned long long* __restrict__ slots, int log2b, int vbits,
              int32_t* __restrict__ status, RowFill fill)
{
    const uint32_t nb = 1u << log2b, nb_mask = nb - 1;
    const uint32_t bound = 5u * nb + 8u;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n;
         r += (int64_t)gridDim.x * blockDim.x) {
        // this row's share of the buffers the probe starts from (coalesced
        // across the warp; hidden behind the insert's round trips)
        for (int q = 0; q < fill.planes; ++q) fill.p[(int64_t)q * fill.stride + r] = -1;
        if (fill.mask) fill.mask[r] = 0u;
        const int4 c = coords[r];
        if (c.x < 0 || c.x >= batch || c.y < 0 || c.y >= D || c.z < 0 || c.z >= H || c.w < 0 ||
            c.w >= W) {
            set_status(status, SPC_ERR_COORD_RANGE);
            continue;
        }
        const unsigned long long key = cell_key(c.x, c.y, c.z, c.w, D, H, W);
        const unsigned long long entry = (key << vbits) | (unsigned long long)r;
        uint32_t bucket = bucket_of(key, log2b);
        // First try the key's home slot in its bucket with a CAS and no read: at
        // load factor <= 1/2 it is usually free, and a taken slot returns its
        // occupant (a duplicate shows here too).  Lookups scan whole buckets, so
        // any free slot of the first non-full bucket is a valid place.
        {
            const unsigned long long old = atomicCAS(&slots[(size_t)bucket * 4 + home_slot(key)], EMPTY, entry);
            if (old == EMPTY) continue;
            if ((old >> vbits) == key) {
                set_status(status, SPC_ERR_DUPLICATE);
                continue;
            }
        }
        uint32_t it = 0;
        for (; it < bound; ++it) {
            unsigned long long v[4];
            load_bucket<true>(slots, bucket, v);
            int empty = -1;
            bool dup = false;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dup |= v[q] != EMPTY && (v[q] >> vbits) == key;
                if (empty < 0 && v[q] == EMPTY) empty = q;
            }
            if (dup) {
                set_status(status, SPC_ERR_DUPLICATE);
                break;
            }
            if (empty < 0) {
                bucket = (bucket + 1) & nb_mask;
                continue;
            }
            const unsigned long long old =
                atomicCAS(&slots[(size_t)bucket * 4 + empty], EMPTY, entry);
            if (old == EMPTY) break;
            if ((old >> vbits) == key) {
                set_status(status, SPC_ERR_DUPLICATE);
                break;
            }
            // another key took that slot first: read the same bucket again
        }
        if (it >= bound) set_status(status, SPC_ERR_TABLE_FULL);
    }
}

// Row of `key`, or -1: resolves the bucket already read in `v`, then walks on.
__device__ __forceinline__ int32_t finish_lookup(const unsigned long long* __restrict__ slots,
                                                 unsigned long long key, uint32_t bucket,
                                                 unsigned long long v[4], int log2b, int vbits,
                                                 int32_t* __restrict__ status)
{
    const unsigned long long vmask = (1ull << vbits) - 1;
    const uint32_t nb = 1u << log2b, nb_mask = nb - 1;
    for (uint32_t it = 0;; ++it) {
        bool empty = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (v[q] != EMPTY && (v[q] >> vbits) == key) return (int32_t)(v[q] & vmask);
            empty |= v[q] == EMPTY;
        }
        if (empty) return -1;
        if (it + 1 >= nb) {
            set_status(status, SPC_ERR_TABLE_FULL);
            return -1;
        }
        bucket = (bucket + 1) & nb_mask;
        load_bucket<false>(slots, bucket, v);
    }
}

// Probe.  A thread owns one output row and a group of kGroup consecutive
// offsets of the probe list; blockIdx.y picks the group, so a warp holds 32
// consecutive rows of one group: coordinates arrive coalesced, map entries
// leave as 128-byte rows of imap, and the group's first buckets are all in
// flight before any is resolved.
//
// MIRROR (submanifold maps): offset k and K-1-k are mirror images (d and -d),
// so imap[K-1-k, i] = o exactly when imap[k, o] = i.  Only k < centre is
// probed; a hit also writes its mirror entry and mirror mask bit, the centre is
// the identity, and the caller has filled imap rows k > centre with -1 and the
// mask with 0 beforehand.
constexpr int kGroup = 2;

// Per-offset table for kernels of at most 32 offsets (precomputed on the host):
// the cell offset of offset k relative to the query's base cell q*stride - pad,
// and the matching difference of cell keys, so a neighbour's key is one add.
constexpr int kMaxTab = 32;
struct ProbeTab {
    int32_t dz[kMaxTab], dy[kMaxTab], dx[kMaxTab];
    long long delta[kMaxTab];
};

template <bool WRITE_T, bool MIRROR>
__global__ void __launch_bounds__(kBlock)
k_map_probe(const int4* __restrict__ q, int64_t nq, int64_t n_in, ProbeGeom g, ProbeTab tab,
            int n_probe, const unsigned long long* __restrict__ slots, int log2b, int vbits,
            int32_t* __restrict__ imap, int32_t* __restrict__ imap_t,
            int32_t* __restrict__ pair_count, uint32_t* __restrict__ mask,
            int32_t* __restrict__ status)
{
    __shared__ int32_t s_cnt[kGroup];
    const int lane = threadIdx.x & 31;
    const int K = g.K;
    const int k0 = blockIdx.y * kGroup;
    if (threadIdx.x < kGroup) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    const int D = g.in_shape[0], H = g.in_shape[1], W = g.in_shape[2];

    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < nq;
         base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = base + threadIdx.x;
        bool valid = r < nq;
        int4 c = make_int4(0, 0, 0, 0);
        if (valid) {
            c = q[r];
            if (c.x < 0 || c.x >= g.batch || c.y < 0 || c.y >= g.q_shape[0] || c.z < 0 ||
                c.z >= g.q_shape[1] || c.w < 0 || c.w >= g.q_shape[2]) {
                if (blockIdx.y == 0) set_status(status, SPC_ERR_COORD_RANGE);
                valid = false;
            }
        }
        const int bz = c.y * g.stride[0] - g.pad[0];
        const int by = c.z * g.stride[1] - g.pad[1];
        const int bx = c.w * g.stride[2] - g.pad[2];
        // key of the (possibly out-of-grid) base cell; in-grid neighbours add delta
        const long long kbase = (((long long)c.x * D + bz) * H + by) * W + bx;

        unsigned long long key[kGroup], v[kGroup][4];
        uint32_t bucket[kGroup];
        bool act[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int k = k0 + u;
            int dz, dy, dx;
            long long dl;
            if (k < kMaxTab) {
                dz = tab.dz[k];
                dy = tab.dy[k];
                dx = tab.dx[k];
                dl = tab.delta[k];
            } else {  // kernels of more than 32 offsets: decode k on the fly
                dz = (k / (g.ksize[1] * g.ksize[2])) * g.dil[0];
                dy = ((k / g.ksize[2]) % g.ksize[1]) * g.dil[1];
                dx = (k % g.ksize[2]) * g.dil[2];
                dl = ((long long)dz * H + dy) * W + dx;
            }
            const int z = bz + dz, y = by + dy, x = bx + dx;
            act[u] = valid && k < n_probe && k != g.centre && (unsigned)z < (unsigned)D &&
                     (unsigned)y < (unsigned)H && (unsigned)x < (unsigned)W;
            key[u] = act[u] ? (unsigned long long)(kbase + dl) : 0ull;
            bucket[u] = bucket_of(key[u], log2b);
            if (act[u]) load_bucket<false>(slots, bucket[u], v[u]);
        }
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int k = k0 + u;
            if (k >= n_probe) break;  // block-uniform
            int32_t row = -1;
            if (act[u]) row = finish_lookup(slots, key[u], bucket[u], v[u], log2b, vbits, status);
            if (valid && k == g.centre) row = (int32_t)r;
            const bool hit = row >= 0;
            if (valid) {
                imap[(int64_t)k * nq + r] = row;
                if (WRITE_T && hit) imap_t[(int64_t)k * n_in + row] = (int32_t)r;
                if (MIRROR && hit && k != g.centre) {
                    imap[(int64_t)(K - 1 - k) * nq + row] = (int32_t)r;
                    if (mask) atomicOr(&mask[row], 1u << ((K - 1 - k) & 31));
                }
            }
            bits |= (hit ? 1u : 0u) << (k & 31);
            const uint32_t hits = __popc(__ballot_sync(FULL_MASK, hit));
            if (lane == 0 && hits) atomicAdd(&s_cnt[u], (int32_t)hits);
        }
        if (mask && valid && bits) atomicOr(&mask[r], bits);
    }
    __syncthreads();
    if (threadIdx.x < kGroup) {
        const int k = k0 + threadIdx.x;
        const int32_t n = s_cnt[threadIdx.x];
        if (k < n_probe && n) {
            atomicAdd(&pair_count[k], n);
            if (MIRROR && k != g.centre) atomicAdd(&pair_count[K - 1 - k], n);
        }
    }
}

// Submanifold 3 x 3 x 3 maps (unit dilation): a thread owns one row and the
// three offsets (dz, dy, -1), (dz, dy, 0), (dz, dy, +1) of one (dz, dy) line
// (blockIdx.y = t < 4: k = 3 t .. 3 t + 2, the lines before the centre's), or
// (t = 4) the offset (0, 0, -1) and the centre.  A warp holds 32 consecutive
// rows; when the previous row is the cell at x - 1 (same sample, z, y), this
// row's (dz, dy, -1) neighbour is that row's (dz, dy, 0) neighbour, found or
// not, and it is taken from the lane below with a shuffle instead of a lookup;
// likewise (dz, dy, +1) from the lane above.  Only the other offsets are looked
// up, all in flight together.  On surface scenes stored in (b, z, y, x) order
// about 60% of rows continue an x-run, so about 40% of the line lookups go.
// The result does not depend on the row order (adjacency is checked on the
// coordinates).  Mirror entries, masks and pair counts as in k_map_probe.
__global__ void __launch_bounds__(kBlock)
k_map_probe_x3(const int4* __restrict__ q, int64_t nq, ProbeGeom g,
               const unsigned long long* __restrict__ slots, int log2b, int vbits,
               int32_t* __restrict__ imap, int32_t* __restrict__ pair_count,
               uint32_t* __restrict__ mask, int32_t* __restrict__ status)
{
    __shared__ int32_t s_cnt[3];
    const int lane = threadIdx.x & 31;
    constexpr int K = 27, kCentre = 13;
    const int t = blockIdx.y;  // 0..3: the line (dz, dy) = (t / 3 - 1, t % 3 - 1); 4: (0, 0, -1) + centre
    const int k0 = 3 * t;
    const int ldz = t < 4 ? t / 3 - 1 : 0, ldy = t < 4 ? t % 3 - 1 : 0;
    if (threadIdx.x < 3) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    const int D = g.in_shape[0], H = g.in_shape[1], W = g.in_shape[2];

    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < nq;
         base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = base + threadIdx.x;
        bool valid = r < nq;
        int4 c = make_int4(-1, -1, -1, -1);
        if (valid) {
            c = q[r];
            if (c.x < 0 || c.x >= g.batch || c.y < 0 || c.y >= D || c.z < 0 || c.z >= H ||
                c.w < 0 || c.w >= W) {
                if (t == 0) set_status(status, SPC_ERR_COORD_RANGE);
                valid = false;
                c = make_int4(-1, -1, -1, -1);
            }
        }
        // the neighbouring lanes' rows: x - 1 below, x + 1 above, same b, z, y
        const int pb = __shfl_up_sync(FULL_MASK, c.x, 1), pz = __shfl_up_sync(FULL_MASK, c.y, 1);
        const int py = __shfl_up_sync(FULL_MASK, c.z, 1), px = __shfl_up_sync(FULL_MASK, c.w, 1);
        const int nb = __shfl_down_sync(FULL_MASK, c.x, 1), nz = __shfl_down_sync(FULL_MASK, c.y, 1);
        const int ny = __shfl_down_sync(FULL_MASK, c.z, 1), nx = __shfl_down_sync(FULL_MASK, c.w, 1);
        const bool adj_prev = valid && lane > 0 && pb == c.x && pz == c.y && py == c.z && px == c.w - 1;
        const bool adj_next = valid && lane < 31 && nb == c.x && nz == c.y && ny == c.z && nx == c.w + 1;
        const long long kbase = (((long long)c.x * D + c.y) * H + c.z) * W + c.w;

        int32_t res[3] = {-1, -1, -1};
        if (t < 4) {
            const int z = c.y + ldz, y = c.z + ldy;
            const bool line_in = valid && (unsigned)z < (unsigned)D && (unsigned)y < (unsigned)H;
            const long long kline = kbase + ((long long)ldz * H + ldy) * W;
            // u = 0: x - 1, 1: x, 2: x + 1; lookups for the centre column and for
            // the side columns the neighbouring lanes cannot supply
            bool act[3];
            unsigned long long key[3], v[3][4];
            uint32_t bucket[3];
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                const int x = c.w + u - 1;
                const bool need = u == 1 || (u == 0 && !adj_prev) || (u == 2 && !adj_next);
                act[u] = line_in && need && (unsigned)x < (unsigned)W;
                key[u] = act[u] ? (unsigned long long)(kline + (u - 1)) : 0ull;
                bucket[u] = bucket_of(key[u], log2b);
                if (act[u]) load_bucket<false>(slots, bucket[u], v[u]);
            }
#pragma unroll
            for (int u = 0; u < 3; ++u)
                if (act[u]) res[u] = finish_lookup(slots, key[u], bucket[u], v[u], log2b, vbits, status);
            const int32_t from_prev = __shfl_up_sync(FULL_MASK, res[1], 1);
            const int32_t from_next = __shfl_down_sync(FULL_MASK, res[1], 1);
            if (adj_prev) res[0] = from_prev;
            if (adj_next) res[2] = from_next;
        } else {
            // (0, 0, -1): the previous row itself when it is the cell at x - 1
            if (adj_prev) {
                res[0] = (int32_t)(r - 1);
            } else if (valid && c.w > 0) {
                const unsigned long long key = (unsigned long long)(kbase - 1);
                const uint32_t bucket = bucket_of(key, log2b);
                unsigned long long v[4];
                load_bucket<false>(slots, bucket, v);
                res[0] = finish_lookup(slots, key, bucket, v, log2b, vbits, status);
            }
            res[1] = valid ? (int32_t)r : -1;  // the centre
        }
        uint32_t bits = 0;
        const int nk = t < 4 ? 3 : 2;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            if (u >= nk) break;  // block-uniform
            const int k = k0 + u;
            const int32_t row = valid ? res[u] : -1;
            const bool hit = row >= 0;
            if (valid) {
                imap[(int64_t)k * nq + r] = row;
                if (hit && k != kCentre) {
                    imap[(int64_t)(K - 1 - k) * nq + row] = (int32_t)r;
                    if (mask) atomicOr(&mask[row], 1u << (K - 1 - k));
                }
            }
            bits |= (hit ? 1u : 0u) << k;
            const uint32_t hits = __popc(__ballot_sync(FULL_MASK, hit));
            if (lane == 0 && hits) atomicAdd(&s_cnt[u], (int32_t)hits);
        }
        if (mask && valid && bits) atomicOr(&mask[r], bits);
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        const int k = k0 + threadIdx.x;
        const int32_t n = s_cnt[threadIdx.x];
        if (threadIdx.x < (t < 4 ? 3 : 2) && n) {
            atomicAdd(&pair_count[k], n);
            if (k != kCentre) atomicAdd(&pair_count[K - 1 - k], n);
        }
    }
}

template <bool WRITE_T, bool MIRROR>
void launch_probe(dim3 grid, cudaStream_t st, const int32_t* qcoords, int64_t nq, int64_t n_in,
                  const ProbeGeom& g, const ProbeTab& tab, int n_probe, HashTable t,
                  int32_t* imap, int32_t* imap_t, int32_t* pair_count, uint32_t* mask,
                  int32_t* status)
{
    k_map_probe<WRITE_T, MIRROR><<<grid, kBlock, 0, st>>>(
        reinterpret_cast<const int4*>(qcoords), nq, n_in, g, tab, n_probe, t.slots,
        t.log2_buckets, t.vbits, imap, imap_t, pair_count, mask, status);
}

}  // namespace

int64_t hash_slots_for(int64_t n)
{
    int64_t s = 64;
    while (s < 2 * n) s <<= 1;
    return s;
}

int hash_vbits_for(int64_t n)
{
    const int b = ceil_log2((uint64_t)(n > 1 ? n : 2));
    return b < 1 ? 1 : b;
}

bool hash_keys_fit(int64_t cells, int vbits)
{
    const int kbits = 64 - vbits;
    if (kbits >= 63) return true;
    return (unsigned long long)cells <= ((1ull << kbits) - 1ull);
}

spc_status build_init(const FillList& L, int n, cudaStream_t st)
{
    int64_t words = 0;
    for (int i = 0; i < n; ++i) words += std::max<int64_t>(L.r[i].n, 0);
    if (n == 0 || words == 0) return SPC_OK;
    FillList l = L;
    for (int i = n; i < 5; ++i) l.r[i] = FillRegion{nullptr, 0, 0u};
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(words / 4 + 30, kBlock), 4 * sm_count()));
    k_build_init<<<grid, kBlock, 0, st>>>(l, n);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

bool probe_mirror(const ProbeGeom& g, bool with_transpose)
{
    return g.centre >= 0 && !with_transpose && g.K == 2 * g.centre + 1;
}

spc_status hash_insert(const int32_t* coords, int64_t n, int32_t batch, const int32_t shape[3],
                       HashTable t, int32_t* status, const RowFill& fill, cudaStream_t st)
{
    if (n == 0) return SPC_OK;
    const int grid = (int)std::min<int64_t>(ceil_div(n, kBlock), 8 * sm_count());
    k_hash_insert<<<grid, kBlock, 0, st>>>(reinterpret_cast<const int4*>(coords), n, batch,
                                           shape[0], shape[1], shape[2], t.slots,
                                           t.log2_buckets, t.vbits, status, fill);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

spc_status map_probe(const int32_t* qcoords, int64_t nq, int64_t n_in, const ProbeGeom& g,
                     HashTable t, int32_t* imap, int32_t* imap_t, int32_t* pair_count,
                     uint32_t* mask, int32_t* status, cudaStream_t st)
{
    if (nq == 0) return SPC_OK;
    // submanifold maps (centre >= 0, odd kernels) are probed for k <= centre only;
    // the caller has zeroed the mask and filled imap rows k > centre with -1
    const bool mirror = probe_mirror(g, imap_t != nullptr);
    const int n_probe = mirror ? g.centre + 1 : g.K;
    ProbeTab tab;
    for (int k = 0; k < kMaxTab; ++k) {
        int dz = 0, dy = 0, dx = 0;
        if (k < g.K) {
            dz = (k / (g.ksize[1] * g.ksize[2])) * g.dil[0];
            dy = ((k / g.ksize[2]) % g.ksize[1]) * g.dil[1];
            dx = (k % g.ksize[2]) * g.dil[2];
        }
        tab.dz[k] = dz;
        tab.dy[k] = dy;
        tab.dx[k] = dx;
        tab.delta[k] = ((long long)dz * g.in_shape[1] + dy) * g.in_shape[2] + dx;
    }
    // submanifold 3 x 3 x 3 maps of unit dilation: x-runs supply the side
    // columns of each line from the neighbouring rows.  Small sets (a few
    // thousand rows: one partial wave, latency-bound) keep the 7 groups of the
    // general probe, which put more threads in flight.
    if (mirror && g.K == 27 && g.centre == 13 && g.ksize[0] == 3 && g.ksize[1] == 3 &&
        g.ksize[2] == 3 && g.dil[0] == 1 && g.dil[1] == 1 && g.dil[2] == 1 && nq >= 4096) {
        const int64_t row_blocks = ceil_div(nq, kBlock);
        const int64_t cap = std::max<int64_t>(1, (int64_t)16 * sm_count() / 5);
        dim3 grid((unsigned)std::min<int64_t>(row_blocks, cap), 5u);
        k_map_probe_x3<<<grid, kBlock, 0, st>>>(reinterpret_cast<const int4*>(qcoords), nq, g, t.slots,
                                                t.log2_buckets, t.vbits, imap, pair_count, mask, status);
        SPC_LAUNCH_CHECK();
        return SPC_OK;
    }
    const int groups = (int)ceil_div(n_probe, kGroup);
    const int64_t row_blocks = ceil_div(nq, kBlock);
    const int64_t cap = std::max<int64_t>(1, (int64_t)16 * sm_count() / groups);
    dim3 grid((unsigned)std::min<int64_t>(row_blocks, cap), (unsigned)groups);
    if (imap_t) launch_probe<true, false>(grid, st, qcoords, nq, n_in, g, tab, n_probe, t, imap, imap_t, pair_count, mask, status);
    else if (mirror) launch_probe<false, true>(grid, st, qcoords, nq, n_in, g, tab, n_probe, t, imap, nullptr, pair_count, mask, status);
    else launch_probe<false, false>(grid, st, qcoords, nq, n_in, g, tab, n_probe, t, imap, nullptr, pair_count, mask, status);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace spc
