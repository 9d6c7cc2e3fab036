// hash.cu -- GPU open-addressing hash table over (b, z, y, x) cell keys and the
// indice-map probe kernel built on it.
//
// Keys: the mixed-radix cell index ((b*D + z)*H + y)*W + x over the grid (the
// int64 key of lato_mlx sparse/conv.py "build_indice_map", here bounded by an
// explicit range check instead of a pad shift).  A slot packs the key above the
// row index, so one 8-byte read both matches and resolves a probe.
//
// Warp-cooperative probing: four lanes own one query and read the four slots of
// one 32-byte bucket together (one L2 sector); a ballot finds a matching key or
// an empty slot.  Inserts claim the first empty slot with a 64-bit CAS.  Every
// probe loop is bounded; exceeding the bound sets SPC_ERR_TABLE_FULL.
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

__device__ __forceinline__ unsigned long long cell_key(int b, int z, int y, int x, int D, int H,
                                                       int W)
{
    return (((unsigned long long)b * D + (unsigned)z) * H + (unsigned)y) * W + (unsigned)x;
}

__global__ void __launch_bounds__(kBlock)
k_hash_clear(unsigned long long* __restrict__ slots, int64_t n)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    ulonglong2* s2 = reinterpret_cast<ulonglong2*>(slots);
    for (; i < n / 2; i += stride) s2[i] = make_ulonglong2(EMPTY, EMPTY);
}

// One key per 4-lane group, eight per warp; the warp stays converged so the
// ballots below always run with the full mask.
__global__ void __launch_bounds__(kBlock)
k_hash_insert(const int4* __restrict__ coords, int64_t n, int32_t batch, int D, int H, int W,
              unsigned long long* __restrict__ slots, int log2b, int vbits,
              int32_t* __restrict__ status)
{
    const int lane = threadIdx.x & 31, sub = lane & 3, gbase = lane & ~3;
    const uint32_t nb = 1u << log2b, nb_mask = nb - 1;
    const uint32_t bound = 5u * nb + 8u;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t wb = warp * 8; wb < n; wb += nwarps * 8) {
        const int64_t r = wb + (lane >> 2);
        bool active = r < n;
        unsigned long long key = 0;
        if (active) {
            const int4 c = coords[r];
            if (c.x < 0 || c.x >= batch || c.y < 0 || c.y >= D || c.z < 0 || c.z >= H ||
                c.w < 0 || c.w >= W) {
                if (sub == 0) set_status(status, SPC_ERR_COORD_RANGE);
                active = false;
            } else {
                key = cell_key(c.x, c.y, c.z, c.w, D, H, W);
            }
        }
        const unsigned long long entry = (key << vbits) | (unsigned long long)r;
        uint32_t bucket = bucket_of(key, log2b);
        for (uint32_t it = 0;; ++it) {
            if (!__any_sync(FULL_MASK, active)) break;
            if (it >= bound) {
                if (active && sub == 0) set_status(status, SPC_ERR_TABLE_FULL);
                break;
            }
            // L2-coherent read: other warps fill slots while this one probes.
            const unsigned long long s = active ? __ldcg(&slots[(size_t)bucket * 4 + sub]) : EMPTY;
            const bool is_match = active && s != EMPTY && (s >> vbits) == key;
            const bool is_empty = active && s == EMPTY;
            const uint32_t gm = (__ballot_sync(FULL_MASK, is_match) >> gbase) & 0xFu;
            const uint32_t ge = (__ballot_sync(FULL_MASK, is_empty) >> gbase) & 0xFu;
            bool won = false;
            if (active && gm == 0 && ge != 0 && sub == __ffs(ge) - 1) {
                const unsigned long long old =
                    atomicCAS(&slots[(size_t)bucket * 4 + sub], EMPTY, entry);
                won = (old == EMPTY);
            }
            const bool group_won = ((__ballot_sync(FULL_MASK, won) >> gbase) & 0xFu) != 0;
            if (active) {
                if (gm != 0) {
                    if (sub == 0) set_status(status, SPC_ERR_DUPLICATE);
                    active = false;
                } else if (group_won) {
                    active = false;
                } else if (ge == 0) {
                    bucket = (bucket + 1) & nb_mask;
                }
                // else: another group took the slot first; read the bucket again
            }
        }
    }
}

// Probe: for each query row r and offset k, the input row at the offset cell.
// ILP: the first bucket of U offsets is loaded before any of them is resolved.
template <bool WRITE_T>
__global__ void __launch_bounds__(kBlock)
k_map_probe(const int4* __restrict__ q, int64_t nq, int64_t n_in, ProbeGeom g,
            const unsigned long long* __restrict__ slots, int log2b, int vbits,
            int32_t* __restrict__ imap, int32_t* __restrict__ imap_t,
            int32_t* __restrict__ pair_count, uint32_t* __restrict__ mask,
            int32_t* __restrict__ status)
{
    constexpr int U = 9;
    extern __shared__ int32_t s_cnt[];  // [K]
    const int lane = threadIdx.x & 31, sub = lane & 3, gbase = lane & ~3;
    const uint32_t nb = 1u << log2b, nb_mask = nb - 1;
    const unsigned long long vmask = (1ull << vbits) - 1;
    const int K = g.K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) s_cnt[k] = 0;
    __syncthreads();

    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int D = g.in_shape[0], H = g.in_shape[1], W = g.in_shape[2];

    for (int64_t wb = warp * 8; wb < nq; wb += nwarps * 8) {
        const int64_t r = wb + (lane >> 2);
        bool valid = r < nq;
        int4 c = make_int4(0, 0, 0, 0);
        if (valid) {
            c = q[r];
            if (c.x < 0 || c.x >= g.batch || c.y < 0 || c.y >= g.q_shape[0] || c.z < 0 ||
                c.z >= g.q_shape[1] || c.w < 0 || c.w >= g.q_shape[2]) {
                if (sub == 0) set_status(status, SPC_ERR_COORD_RANGE);
                valid = false;
            }
        }
        const int bz = c.y * g.stride[0] - g.pad[0];
        const int by = c.z * g.stride[1] - g.pad[1];
        const int bx = c.w * g.stride[2] - g.pad[2];
        uint32_t m = 0;

        for (int k0 = 0; k0 < K; k0 += U) {
            unsigned long long key[U], s[U];
            uint32_t bucket[U];
            bool act[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u;
                act[u] = false;
                key[u] = 0;
                bucket[u] = 0;
                s[u] = EMPTY;
                if (k < K && valid && k != g.centre) {
                    const int kx = k % g.ksize[2];
                    const int ky = (k / g.ksize[2]) % g.ksize[1];
                    const int kz = k / (g.ksize[2] * g.ksize[1]);
                    const int z = bz + kz * g.dil[0], y = by + ky * g.dil[1], x = bx + kx * g.dil[2];
                    if (z >= 0 && z < D && y >= 0 && y < H && x >= 0 && x < W) {
                        act[u] = true;
                        key[u] = cell_key(c.x, z, y, x, D, H, W);
                        bucket[u] = bucket_of(key[u], log2b);
                        s[u] = __ldg(&slots[(size_t)bucket[u] * 4 + sub]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u;
                if (k >= K) break;  // warp-uniform
                int32_t row = -1;
                bool active = act[u];
                unsigned long long sv = s[u];
                for (uint32_t it = 0;; ++it) {
                    const bool is_match = active && sv != EMPTY && (sv >> vbits) == key[u];
                    const bool is_empty = active && sv == EMPTY;
                    const uint32_t bm = __ballot_sync(FULL_MASK, is_match);
                    const uint32_t be = __ballot_sync(FULL_MASK, is_empty);
                    const uint32_t gm = (bm >> gbase) & 0xFu, ge = (be >> gbase) & 0xFu;
                    const int src = gm ? gbase + __ffs(gm) - 1 : lane;
                    const unsigned long long hit = __shfl_sync(FULL_MASK, sv, src);
                    if (active) {
                        if (gm) {
                            row = (int32_t)(hit & vmask);
                            active = false;
                        } else if (ge) {
                            active = false;
                        } else if (it + 1 >= nb) {
                            if (sub == 0) set_status(status, SPC_ERR_TABLE_FULL);
                            active = false;
                        } else {
                            bucket[u] = (bucket[u] + 1) & nb_mask;
                        }
                    }
                    if (!__any_sync(FULL_MASK, active)) break;
                    sv = active ? __ldg(&slots[(size_t)bucket[u] * 4 + sub]) : EMPTY;
                }
                if (valid && k == g.centre) row = (int32_t)r;
                const bool hitb = row >= 0;
                if (sub == 0 && valid) {
                    imap[(int64_t)k * nq + r] = row;
                    if (WRITE_T && hitb) imap_t[(int64_t)k * n_in + row] = (int32_t)r;
                }
                m |= (hitb ? 1u : 0u) << (k & 31);
                const uint32_t hits = __popc(__ballot_sync(FULL_MASK, sub == 0 && hitb));
                if (lane == 0 && hits) atomicAdd(&s_cnt[k], (int32_t)hits);
            }
        }
        if (mask && sub == 0 && valid) mask[r] = m;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += blockDim.x)
        if (s_cnt[k]) atomicAdd(&pair_count[k], s_cnt[k]);
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

spc_status hash_clear(HashTable t, cudaStream_t st)
{
    const int64_t n = 4ll << t.log2_buckets;
    const int grid = (int)std::min<int64_t>(ceil_div(n / 2, kBlock), 4 * sm_count());
    k_hash_clear<<<grid, kBlock, 0, st>>>(t.slots, n);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

spc_status hash_insert(const int32_t* coords, int64_t n, int32_t batch, const int32_t shape[3],
                       HashTable t, int32_t* status, cudaStream_t st)
{
    if (n == 0) return SPC_OK;
    const int64_t warps = ceil_div(n, 8);
    const int grid = (int)std::min<int64_t>(ceil_div(warps * 32, kBlock), 16 * sm_count());
    k_hash_insert<<<grid, kBlock, 0, st>>>(reinterpret_cast<const int4*>(coords), n, batch,
                                           shape[0], shape[1], shape[2], t.slots,
                                           t.log2_buckets, t.vbits, status);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

spc_status map_probe(const int32_t* qcoords, int64_t nq, int64_t n_in, const ProbeGeom& g,
                     HashTable t, int32_t* imap, int32_t* imap_t, int32_t* pair_count,
                     uint32_t* mask, int32_t* status, cudaStream_t st)
{
    if (nq == 0) return SPC_OK;
    const int64_t warps = ceil_div(nq, 8);
    const int grid = (int)std::min<int64_t>(ceil_div(warps * 32, kBlock), 16 * sm_count());
    const size_t smem = sizeof(int32_t) * (size_t)g.K;
    if (imap_t) {
        k_map_probe<true><<<grid, kBlock, smem, st>>>(
            reinterpret_cast<const int4*>(qcoords), nq, n_in, g, t.slots, t.log2_buckets, t.vbits,
            imap, imap_t, pair_count, mask, status);
    } else {
        k_map_probe<false><<<grid, kBlock, smem, st>>>(
            reinterpret_cast<const int4*>(qcoords), nq, n_in, g, t.slots, t.log2_buckets, t.vbits,
            imap, nullptr, pair_count, mask, status);
    }
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace spc
