// conv_tile.cuh -- the prologue every gathered tensor-core conv tile runs:
// which map entries the tile's rows need, and which offsets the tile uses.
#pragma once

#include "common.cuh"

namespace spc {

// A tile's view of the map: tile row r computes output row perm[r] (or
// row0 + r), whose neighbour through offset k is map[mk * rows + row] with mk
// = k, or K - 1 - k for a mirrored submanifold map; map == NULL is the
// identity (K == 1).  mask (with perm) holds each row's offset bits.
struct TileMap {
    const int32_t* map;
    const uint32_t* mask;
    const int32_t* perm;
    int64_t rows, in_rows;
    int32_t K, mirror;
};

// Fills s_idx[a * kRows + r] with the input row of tile row r through the
// tile's a-th active offset (-1 for none) and s_active[a] with that offset;
// returns the number of active offsets.  Threads tid < kRows own one tile row
// each; every thread of the block must call this (it holds __syncthreads).
// s_union must be 0 on entry (set before a barrier).
//
// Rows in a caller's grouped order (perm and mask given) have few offsets
// each: their masks are read first and only those entries are loaded.
// Otherwise all K entries of a row are loaded in one burst (no dependent mask
// read first) and the tile's offsets are those where some row has an entry.
template <int kRows>
__device__ __forceinline__ int tile_map_entries(const TileMap& t, int64_t row0, int tid,
                                                int32_t* s_idx, int* s_active, int* s_nact,
                                                unsigned* s_union)
{
    const int lane = tid & 31;
    const uint32_t kmask = t.K >= 32 ? 0xffffffffu : ((1u << t.K) - 1u);
    const bool rvalid = tid < kRows && row0 + tid < t.rows;
    const int64_t row = rvalid && t.perm ? (int64_t)__ldg(t.perm + row0 + tid) : row0 + tid;
    const bool by_mask = t.perm && t.mask;
    int32_t iv[32];
    uint32_t m = 0;
    if (tid < kRows) {
        if (by_mask) {
            if (rvalid) {
                m = __ldcs(t.mask + row);  // read once: evict first
                if (t.mirror) m = __brev(m) >> (32 - t.K);
                m &= kmask;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                iv[k] = -1;
                if (k < t.K && rvalid) {
                    const int mk = t.mirror ? t.K - 1 - k : k;
                    iv[k] = t.map ? __ldcs(t.map + (int64_t)mk * t.rows + row) : (int32_t)row;
                }
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                if (iv[k] >= t.in_rows || iv[k] < 0) iv[k] = -1;
                m |= (iv[k] >= 0 ? 1u : 0u) << k;
            }
        }
        const uint32_t wu = __reduce_or_sync(FULL_MASK, m);
        if (lane == 0 && wu) atomicOr(s_union, wu);
    }
    __syncthreads();
    const uint32_t uni = *s_union;
    if (tid == 0) {
        uint32_t u = uni;
        int n = 0;
        while (u) {
            s_active[n++] = __ffs(u) - 1;
            u &= u - 1;
        }
        *s_nact = n;
    }
    if (tid < kRows && !by_mask) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if ((uni >> k) & 1u) s_idx[__popc(uni & ((1u << k) - 1u)) * kRows + tid] = iv[k];
    }
    __syncthreads();
    const int nact = *s_nact;
    if (by_mask) {
        if (tid < kRows) {
            // this row's entries for the tile's active offsets, all loads in flight
            // before the first store
#pragma unroll
            for (int ai = 0; ai < 32; ++ai) {
                iv[ai] = -1;
                if (ai < nact) {
                    const int k = s_active[ai];
                    if (rvalid && ((m >> k) & 1u)) {
                        const int mk = t.mirror ? t.K - 1 - k : k;
                        iv[ai] = __ldcs(t.map + (int64_t)mk * t.rows + row);
                    }
                }
            }
#pragma unroll
            for (int ai = 0; ai < 32; ++ai)
                if (ai < nact) s_idx[ai * kRows + tid] = (iv[ai] >= 0 && iv[ai] < t.in_rows) ? iv[ai] : -1;
        }
        __syncthreads();
    }
    return nact;
}

}  // namespace spc
