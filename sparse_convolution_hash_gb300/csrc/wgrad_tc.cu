// wgrad_tc.cu -- dfilter on the tcgen05 tensor cores:
//   dW[k][c][j] = sum over output rows o with i = imap[k, o] != -1 of x[i][c] dy[o][j].
//
// Each CTA owns a group of up to 8 kernel offsets, one 64 x 64 tile of dW
// (input-channel block x output-channel block) and a fixed chunk of output
// rows.  For every 128-row slice of its chunk it loads the dy rows once (one
// 2-D TMA load, 128 x 128 bytes) and gathers the matching x rows of each of its
// offsets through the map with cp.async (rows without a pair are zero-filled,
// so they add nothing).  The reduction runs over rows, so both operands are
// MN-major: a gathered row is 64 channels (the M index) of one reduction
// index.  Offsets go in pairs: the two offsets' gathered rows are the two
// 64-channel atoms of one M = 128 operand, so one MMA (M = 128, N = 64, K = 16
// rows) accumulates both offsets' 64 x 64 tiles at once, in lanes 0-63 and
// 64-127 of 64 tensor-memory columns (an odd offset out runs as M = 64).  Four
// pairs take 256 columns, half of an SM's 512, so two CTAs share an SM and one's
// waits overlap the other's gathers.  At the end the CTA writes its partial
// tiles to the workspace; k_wgrad_reduce sums the chunks in a fixed order, so
// dW is run-to-run bit-identical.
//
// Every wait is bounded.  The waits of one warp role on another give up after
// the library's wait limit (spc_set_wait_limit_ns, 2 s by default) and set
// SPC_ERR_TIMEOUT; the CTA then waits for the copies and MMAs it issued itself
// (bounded by 2 s: those always complete), frees its tensor memory and returns.
#include "kernels.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace spc {

namespace {

constexpr int kRows = 128;      // reduction rows per slice
constexpr int kGroup = 8;       // offsets per CTA
constexpr int kPairs = kGroup / 2;
constexpr int kStages = 2;      // x-gather stages, one offset pair (two 16 KB atoms) each
constexpr int kWorkers = 256;   // warps 0-7: gathers (eight 16-byte copies each per stage); warps 0-3 then run the epilogue
constexpr int kThreads = kWorkers + 64;  // warp 8: dy TMA; warp 9: TMEM owner, MMA issuer
constexpr int kTmaWarp = kWorkers / 32, kMmaWarp = kTmaWarp + 1;
constexpr uint64_t kDrainNs = 2000000000ull;  // bound of the waits for a CTA's own copies / MMAs
constexpr int kAtomBytes = kRows * 128;  // 128 rows x 64 channels x 2 bytes: one offset's rows
constexpr int kABytes = 2 * kAtomBytes;  // a pair stage
constexpr int kBBytes = kRows * 128;
constexpr int kTmemCols = kPairs * 64;
constexpr int kMapPer = kGroup * kRows / kWorkers;  // map entries each gather thread stages per slice

template <typename T> struct TcKindW;
template <> struct TcKindW<__half> { static constexpr uint32_t fmt = 0; };
template <> struct TcKindW<__nv_bfloat16> { static constexpr uint32_t fmt = 1; };

// About 106 KB: two CTAs fit in an SM's shared memory (and its tensor memory).
size_t smem_bytes()
{
    return 1024 + (size_t)kStages * kABytes + 2 * (size_t)kBBytes + 2 * kGroup * kRows * 4 +
           8 * (2 * kStages + 5) + 64;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
k_wgrad_tc(WgradTcArgs a, const __grid_constant__ CUtensorMap tma_dy)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* As = smem;                               // [kStages][2 atoms][kAtomBytes]
    uint8_t* Bs = smem + (size_t)kStages * kABytes;   // [2][kBBytes]
    int32_t* s_map = reinterpret_cast<int32_t*>(Bs + 2 * (size_t)kBBytes);  // [2][kGroup][kRows]
    uint64_t* afull = reinterpret_cast<uint64_t*>(s_map + 2 * kGroup * kRows);
    uint64_t* aempty = afull + kStages;
    uint64_t* bfull = aempty + kStages;
    uint64_t* bempty = bfull + 2;
    uint64_t* done = bempty + 2;
    int* s_ctrl = reinterpret_cast<int*>(done + 1);  // abort, tmem
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // which offsets, which dW tile, which rows
    const int tiles_c = a.cin / 64, tiles_j = a.cout / 64;
    int t = blockIdx.x;
    const int jt = t % tiles_j;
    t /= tiles_j;
    const int ct = t % tiles_c;
    const int kg = t / tiles_c;
    // the K offsets are split into ceil(K / kGroup) groups of near-equal size
    // (27 -> 7, 7, 7, 6), so every CTA of a row split does about the same work
    const int n_groups = (a.K + kGroup - 1) / kGroup;
    const int g_base = a.K / n_groups, g_rem = a.K % n_groups;
    const int k0 = kg * g_base + (kg < g_rem ? kg : g_rem);
    const int ng = g_base + (kg < g_rem ? 1 : 0);
    const int np = (ng + 1) / 2;  // pairs, the last one single when ng is odd
    const int s_split = blockIdx.y;
    const int64_t o_lo = (int64_t)s_split * a.chunk;
    const int64_t o_hi = o_lo + a.chunk < a.n_out ? o_lo + a.chunk : a.n_out;
    const int nrc = o_hi > o_lo ? (int)((o_hi - o_lo + kRows - 1) / kRows) : 0;
    const int n_iter = nrc * np;
    const int c0 = ct * 64, j0 = jt * 64;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&afull[s], kWorkers);
            ptx::mbar_init(&aempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bfull[b], 1);
            ptx::mbar_init(&bempty[b], 1);
        }
        ptx::mbar_init(done, 1);
        s_ctrl[0] = 0;
        ptx::mbar_init_fence();
    }
    if (warp == kTmaWarp && lane == 0) ptx::prefetch_tmap(&tma_dy);
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&s_ctrl[1]), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = (uint32_t)s_ctrl[1];

    if (tid < kWorkers) {
        // ------------------------------------------------------ x-row gathers
        // thread t copies 16-byte chunk (t & 7) of rows 32 j + t / 8 (j < 4) of
        // each atom.  The map entries of the next 128-row slice (all offsets of
        // the group) are read into registers while the current slice is issued
        // and staged in shared memory behind one barrier of the gather warps per
        // slice, so no copy waits on a map read.
        const uint8_t* x = static_cast<const uint8_t*>(a.x);
        const uint64_t keep = ptx::policy_evict_last();
        const int ch = tid & 7;
        auto load_map = [&](int rc, int32_t (&v)[kMapPer]) {
#pragma unroll
            for (int q = 0; q < kMapPer; ++q) {
                const int e = q * kWorkers + tid;  // entry (offset g, row r) of the slice
                const int g = e / kRows, r = e % kRows;
                const int64_t o = o_lo + (int64_t)rc * kRows + r;
                int32_t i = -1;
                if (g < ng && rc < nrc && o < o_hi) i = __ldg(a.map + (int64_t)(k0 + g) * a.n_out + o);
                v[q] = (i >= 0 && i < a.n_in) ? i : -1;
            }
        };
        auto store_map = [&](int rc, const int32_t (&v)[kMapPer]) {
#pragma unroll
            for (int q = 0; q < kMapPer; ++q) s_map[(rc & 1) * kGroup * kRows + q * kWorkers + tid] = v[q];
        };
        int32_t nxt[kMapPer];
        load_map(0, nxt);
        store_map(0, nxt);
        ptx::bar_sync_named(1, kWorkers);
        for (int rc = 0; rc < nrc; ++rc) {
            load_map(rc + 1, nxt);
            const int32_t* m = s_map + (rc & 1) * kGroup * kRows;
            for (int p = 0; p < np; ++p) {
                const int it = rc * np + p;
                const int s = it % kStages;
                if (it >= kStages && !ptx::mbar_wait(&aempty[s], ((it / kStages) - 1) & 1, a.wait_ns)) {
                    atomicExch(&s_ctrl[0], 1);
                    break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int g = 2 * p + h;
                    if (g >= ng) break;
                    const uint32_t abase = ptx::smem_u32(As + (size_t)s * kABytes + (size_t)h * kAtomBytes);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = j * (kWorkers / 8) + (tid >> 3);
                        const int32_t i = m[g * kRows + r];
                        const uint8_t* src = i >= 0 ? x + ((int64_t)i * a.cin + c0) * sizeof(T) + ch * 16 : x;
                        ptx::cp_async16_hint(abase + (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4),
                                             src, i >= 0 ? 16u : 0u, keep);
                    }
                }
                ptx::cp_async_arrive_noinc(&afull[s]);
            }
            store_map(rc + 1, nxt);
            // every gather thread reaches this barrier (a thread whose wait ran
            // out skips the rest of its slice), so the abort flag is seen by all
            ptx::bar_sync_named(1, kWorkers);
            if (s_ctrl[0]) break;
        }
        ptx::cp_async_wait_all();
    } else if (warp == kTmaWarp) {
        // --------------------------------------------------- dy rows (TMA)
        if (lane == 0) {
            int issued = 0;
            for (int rc = 0; rc < nrc; ++rc) {
                const int b = rc & 1;
                if (rc >= 2 && !ptx::mbar_wait(&bempty[b], ((rc >> 1) - 1) & 1, a.wait_ns)) {
                    atomicExch(&s_ctrl[0], 1);
                    break;
                }
                ptx::mbar_arrive_expect_tx(&bfull[b], kBBytes);
                ptx::tma_tile2d(ptx::smem_u32(Bs + (size_t)b * kBBytes), &tma_dy, j0,
                                (int32_t)(o_lo + (int64_t)rc * kRows), &bfull[b]);
                ++issued;
            }
            const int first = issued > 2 ? issued - 2 : 0;
            for (int rc = first; rc < issued; ++rc) ptx::mbar_wait(&bfull[rc & 1], (rc >> 1) & 1, kDrainNs);
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        // M = 128 (two offsets' 64 input channels) or 64 (one), N = 64 output
        // channels, both operands MN-major
        const uint32_t mn = (1u << 15) | (1u << 16);
        const uint32_t idesc2 = ptx::idesc_make(TcKindW<T>::fmt, 128, 64) | mn;
        const uint32_t idesc1 = ptx::idesc_make(TcKindW<T>::fmt, 64, 64) | mn;
        bool ok = true;
        for (int rc = 0; rc < nrc && ok; ++rc) {
            const int b = rc & 1;
            if (!ptx::mbar_wait(&bfull[b], (rc >> 1) & 1, a.wait_ns)) {
                ok = false;
                break;
            }
            const uint32_t bbase = ptx::smem_u32(Bs + (size_t)b * kBBytes);
            for (int p = 0; p < np; ++p) {
                const int it = rc * np + p;
                const int s = it % kStages;
                if (!ptx::mbar_wait(&afull[s], (it / kStages) & 1, a.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::fence_proxy_async_smem();  // the x rows arrived through generic-proxy copies
                ptx::tc_fence_after();
                const uint32_t abase = ptx::smem_u32(As + (size_t)s * kABytes);
                const uint32_t idesc = 2 * p + 1 < ng ? idesc2 : idesc1;
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)  // 16 reduction rows (two 8-row groups) per instruction
                    // A: two 64-channel atoms kAtomBytes apart; B one atom wide
                    ptx::mma<0>(tmem + (uint32_t)(p * 64), ptx::desc_mn_sw128(abase + kk * 2048, kAtomBytes),
                                ptx::desc_mn_sw128(bbase + kk * 2048, 16), idesc,
                                (rc | kk) != 0 ? 1u : 0u);
                ptx::mma_commit(&aempty[s]);
            }
            ptx::mma_commit(&bempty[b]);
        }
        if (!ok) atomicExch(&s_ctrl[0], 1);
        ptx::mma_commit(done);
    }

    // ------------------------------------------------------------ epilogue
    // A pair's M = 128 accumulator rows sit in TMEM lanes 0-127: warp q of the
    // first four holds rows 32 q .. 32 q + 31 (rows 0-63: the pair's first
    // offset, 64-127 its second).  A single offset's M = 64 rows sit in lanes
    // 32 q + r (r < 16): warp q holds rows 16 q .. 16 q + 15 in lanes 0-15.
    if (warp < 4) {
        const bool waited = ptx::mbar_wait(done, 0, kDrainNs);
        ptx::tc_fence_after();
        const bool aborted = __any_sync(FULL_MASK, !waited || s_ctrl[0] != 0);
        if (aborted) {
            if (tid == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        } else {
            for (int p = 0; p < np; ++p) {
                const bool pair = 2 * p + 1 < ng;
                const int m = pair ? warp * 32 + lane : warp * 16 + lane;  // accumulator row
                const int g = 2 * p + (pair ? m / 64 : 0);
                const int c = m % 64;                                     // input channel within the tile
                const bool active = pair || lane < 16;
                const int tile = ((k0 + g) * tiles_c + ct) * tiles_j + jt;
                float* dst = a.part + ((size_t)tile * a.splits + s_split) * 4096 + (size_t)c * 64;
#pragma unroll 1
                for (int cc = 0; cc < 64; cc += 32) {
                    uint32_t v[32];
                    if (n_iter > 0) {
                        ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(p * 64 + cc), v);
                        ptx::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0u;
                    }
                    if (active) {
                        float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            d4[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename T>
spc_status launch(const WgradTcArgs& a, cudaStream_t st)
{
    CUtensorMap tdy;
    const CUtensorMapDataType dtt = TcKindW<T>::fmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!tmap_2d(&tdy, dtt, 2, a.dy, (uint64_t)a.cout, (uint64_t)a.n_out, 64, kRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
        return SPC_ERR_UNSUPPORTED;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPC_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(k_wgrad_tc<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes()) != cudaSuccess)
            return SPC_ERR_UNSUPPORTED;
        configured[dev] = true;
    }
    const int groups = (a.K + kGroup - 1) / kGroup;
    dim3 grid((unsigned)(groups * (a.cin / 64) * (a.cout / 64)), (unsigned)a.splits);
    k_wgrad_tc<T><<<grid, kThreads, smem_bytes(), st>>>(a, tdy);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace

bool wgrad_tc_supported(int32_t K, int32_t cin, int32_t cout, spc_dtype dt)
{
    return (dt == SPC_F16 || dt == SPC_BF16) && K >= 1 && cin % 64 == 0 && cout % 64 == 0;
}

// Row splits: at most two CTAs per SM of a 152-SM GB300 (a CTA takes half of its
// SM's tensor memory, so more CTAs than that would wait for a second wave).  A
// fixed target (not the device's SM count) keeps the summation order, and so
// the result bits, the same on every device.
int wgrad_tc_splits(int32_t K, int64_t n_out, int32_t cin, int32_t cout)
{
    constexpr int64_t kTargetCtas = 304;
    const int64_t tiles = (int64_t)((K + kGroup - 1) / kGroup) * (cin / 64) * (cout / 64);
    int64_t s = tiles > 0 ? kTargetCtas / tiles : 1;
    const int64_t max_s = n_out > 0 ? (n_out + kRows - 1) / kRows : 1;
    if (s > max_s) s = max_s;
    return (int)(s < 1 ? 1 : s);
}

spc_status wgrad_tc(const WgradTcArgs& a, spc_dtype dt, cudaStream_t st)
{
    switch (dt) {
    case SPC_F16: return launch<__half>(a, st);
    case SPC_BF16: return launch<__nv_bfloat16>(a, st);
    default: return SPC_ERR_UNSUPPORTED;
    }
}

}  // namespace spc
