// conv_tc.cu -- gathered implicit GEMM on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory) for wide channels.
//
// Output-stationary: a CTA owns MT x 128 output rows (MT 128-row MMA tiles with
// their own accumulators, sharing every weight stage) x BN output channels.  It
// reads its rows' map entries in one burst and skips the offsets no row of the
// tile uses (rows in a caller's grouped order read their masks first and load
// only the entries they have).  The K loop then runs over (active offset, 128-byte channel chunk):
//   NW gather warps copy the tile's input rows of that offset with 16-byte
//     cp.async copies straight into a 128-byte-swizzled K-major shared-memory
//     stage (a warp instruction copies four whole 128-byte row segments; rows
//     with no neighbour are zero-filled by the copy itself); each thread's
//     copies arrive on the stage's mbarrier when they land, so no thread waits
//     for its own data;
//   one thread of warp NW loads the BN x 128-byte weight tile with a 2-D TMA
//     load that completes on the same barrier;
//   one thread of warp NW + 1 waits for the stage, fences the copies into the
//     async proxy, issues MT x 4 tcgen05.mma (one per 128-row tile, K = 32
//     bytes each) into the fp32 accumulators in tensor memory, and commits
//     the stage back to the producers.
// Shapes with 8 gather warps run two CTAs per SM, so one CTA's map-entry burst
// and epilogue overlap the other's gathers.
// All offsets accumulate in tensor memory; the epilogue (the gather warps) reads each
// row's accumulators with tcgen05.ld, adds the bias, rounds once and, for rows in
// tile order, stages the tile in the freed stage buffers as 128-byte-swizzled
// boxes that one thread stores with 2-D TMA (rows in a caller's order are
// stored by their threads).  Every output row is written once: no atomics,
// run-to-run identical.
//
// Forward: B = W[k] as stored, [Cin][Cout], read as an MN-major operand (K =
// Cin rows of N = Cout contiguous channels), loaded with 2-D TMA boxes of 64
// rows x 64 channels; the 16- and 32-channel row shapes and tf32 take the
// weights transposed to [Cout][Cin] (K-major) in the workspace instead.
// dinput: rows are input rows, the map is the transposed or mirrored map, and
// B = W[k] as stored ([Cin][Cout] is already [N][K] K-major for that product).
//
// Every wait is bounded.  The waits of one warp role on another (a free stage,
// a full stage) give up after the library's wait limit (spc_set_wait_limit_ns,
// 2 s by default); a wait that runs out sets SPC_ERR_TIMEOUT in the status
// word, and the CTA then waits for the copies and MMAs it issued itself (bounded
// by 2 s: those always complete), frees its tensor memory and returns.
#include "conv_tile.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace spc {

namespace {

constexpr int kHalf = 128;  // rows per MMA (M)
#ifndef TC_MT
#define TC_MT 2
#endif
#ifndef TC_NW
#define TC_NW 16
#endif
#ifndef TC_STAGES
#define TC_STAGES 4
#endif
// shape of the narrow-row (16 / 32 channel) instances
#ifndef TCN_MT
#define TCN_MT 1
#endif
#ifndef TCN_NW
#define TCN_NW 4
#endif
#ifndef TCN_STAGES
#define TCN_STAGES 8
#endif
constexpr uint64_t kDrainNs = 2000000000ull;  // bound of the waits for a CTA's own copies / MMAs

// MT 128-row MMA tiles per CTA share every weight stage (MT accumulators in
// TMEM); NW warps gather rows and later run the epilogue; warp NW issues the
// weight TMA and warp NW + 1 owns TMEM and issues the MMAs.
template <typename T, int BN, int STAGES, int MT, int NW, int RB>
struct TcShape {
    static constexpr int kRowsPerCta = MT * kHalf;
    static constexpr int kWorkers = NW * 32;
    static constexpr int kThreads = kWorkers + 64;
    static constexpr int kTmaWarp = NW, kMmaWarp = NW + 1;
    static constexpr int ELEM = (int)sizeof(T);
    static constexpr int CH = RB / ELEM;   // elements per RB-byte chunk of a row
    static constexpr int CPR = RB / 16;    // 16-byte pieces per row chunk
    static constexpr int A_BYTES = kRowsPerCta * RB;
    static constexpr int B_BYTES = BN * RB;
    static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + 1023) / 1024 * 1024;
    static constexpr int TMEM_COLS = MT * BN <= 32 ? 32 : (MT * BN <= 64 ? 64 : (MT * BN <= 128 ? 128 : (MT * BN <= 256 ? 256 : 512)));
    // shapes of at most 8 gather warps are built to share an SM with a second CTA
    static constexpr int kMinCtas = (MT == 1 || NW <= 8) ? 2 : 1;
    // The epilogue can stage the tile's output (rows x BN) in the freed stage
    // buffers as 128-row x 128-byte boxes and store them with TMA.
    static constexpr bool kTmaStore =
        (BN * ELEM) % 128 == 0 && (size_t)kRowsPerCta * BN * ELEM <= (size_t)STAGES * STAGE_BYTES;
    static size_t smem_bytes(int K)
    {
        return 1024 /* alignment slack */ + (size_t)STAGES * STAGE_BYTES +
               (size_t)K * kRowsPerCta * 4 + 8 * (2 * STAGES + 1) + 4 * 40;
    }
};

template <typename T> struct TcKind;
template <> struct TcKind<__half> { static constexpr int kind = 0; static constexpr uint32_t fmt = 0; };
template <> struct TcKind<__nv_bfloat16> { static constexpr int kind = 0; static constexpr uint32_t fmt = 1; };
template <> struct TcKind<float> { static constexpr int kind = 1; static constexpr uint32_t fmt = 2; };

// DENSE: K == 1 on the identity map (a per-voxel GEMM): the A tiles are whole
// row blocks of the input, loaded with 2-D TMA like the weights (no gathers,
// no map entries); the gather warps only run the epilogue.
template <typename T, int BN, int STAGES, int MT, int NW, int RB, bool BMN, bool DENSE>
__global__ void __launch_bounds__(TcShape<T, BN, STAGES, MT, NW, RB>::kThreads, TcShape<T, BN, STAGES, MT, NW, RB>::kMinCtas)
k_conv_tc(TcArgs a, const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ CUtensorMap tma_o,
          const __grid_constant__ CUtensorMap tma_a, int tstore)
{
    using S = TcShape<T, BN, STAGES, MT, NW, RB>;
    constexpr int kRowsPerCta = S::kRowsPerCta, kWorkers = S::kWorkers;
    constexpr int kTmaWarp = S::kTmaWarp, kMmaWarp = S::kMmaWarp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int K = a.K;
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + (size_t)STAGES * S::STAGE_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(s_idx + (size_t)K * kRowsPerCta);
    uint64_t* empty = full + STAGES;
    uint64_t* done = empty + STAGES;
    int* s_active = reinterpret_cast<int*>(done + 1);  // [32]
    int* s_ctrl = s_active + 32;                      // nact, abort, union, tmem
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
    const int n0 = blockIdx.y * BN;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // one copy completion per worker + the weight TMA (dense: the TMA alone)
            ptx::mbar_init(&full[s], DENSE ? 1 : kWorkers + 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        s_ctrl[0] = 0;
        s_ctrl[1] = 0;
        s_ctrl[2] = 0;
        ptx::mbar_init_fence();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tmap(&tma_b);
        if (DENSE) ptx::prefetch_tmap(&tma_a);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&s_ctrl[3]), S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // the tile's map entries (thread t owns row t of the tile) and active offsets
    int nact = 1;
    if constexpr (DENSE) {
        if (tid == 0) s_active[0] = 0;
        __syncthreads();
    } else {
        const TileMap tm{a.map, a.mask, a.perm, a.rows, a.in_rows, a.K, a.mirror};
        nact = tile_map_entries<kRowsPerCta>(tm, row0, tid, s_idx, s_active, &s_ctrl[0],
                                             reinterpret_cast<unsigned*>(&s_ctrl[2]));
    }
    const int kchunks = a.cred / S::CH;
    const int n_iter = nact * kchunks;
    const uint32_t tmem = (uint32_t)s_ctrl[3];

    const uint8_t* in = static_cast<const uint8_t*>(a.in);
    if (tid < kWorkers) {
        if constexpr (!DENSE) {
        // -------------------------------------------------- row-gather producers
        // A stage: the tile's rows x RB / 16 chunks of 16 bytes; chunk e = j *
        // kWorkers + tid, so a warp instruction copies whole row segments (four
        // of 128 bytes).  The gather warps of the SM's CTAs (16 per SM) keep
        // enough copies in flight to cover L2 latency.  Each thread's copies
        // arrive on the stage's barrier when they complete, so the thread never
        // waits for its own data, only for a free stage.
        // feature rows are re-read by up to K output rows: keep them in L2
        const uint64_t keep = ptx::policy_evict_last();
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            bool ok = true;
            if (it >= STAGES) ok = ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, a.wait_ns);
            if (!ok) {
                atomicExch(&s_ctrl[1], 1);
                break;
            }
            const int ai = it / kchunks;
            const int c0 = (it % kchunks) * S::CH;
            const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
            const int32_t* idx = s_idx + ai * kRowsPerCta;
#pragma unroll
            for (int j = 0; j < (kRowsPerCta * S::CPR + kWorkers - 1) / kWorkers; ++j) {
                const int e = j * kWorkers + tid;
                if (e >= kRowsPerCta * S::CPR) break;
                const int r = e / S::CPR, ch = e % S::CPR;
                // RB-byte swizzle: the piece index XORs with bits 7.. of the row's offset
                const int sw = ((r * RB) >> 7) & (S::CPR - 1);
                const int32_t i = idx[r];
                const uint8_t* src = i >= 0 ? in + ((int64_t)i * a.cred + c0) * S::ELEM + ch * 16 : in;
                ptx::cp_async16_hint(a_base + (uint32_t)r * RB + ((uint32_t)(ch ^ sw) << 4), src,
                                     i >= 0 ? 16u : 0u, keep);
            }
            ptx::cp_async_arrive_noinc(&full[s]);
        }
        ptx::cp_async_wait_all();  // nothing of ours may still land when the CTA ends
        }
    } else if (warp == kTmaWarp) {
        // -------------------------------------------------- weight producer (TMA)
        int issued = 0;
        if (lane == 0) {
            for (int it = 0; it < n_iter; ++it) {
                const int s = it % STAGES;
                if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, a.wait_ns)) {
                    atomicExch(&s_ctrl[1], 1);
                    break;
                }
                const int ai = it / kchunks;
                const int c0 = (it % kchunks) * S::CH;
                const int k = s_active[ai];
                const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
                ptx::mbar_arrive_expect_tx(&full[s], DENSE ? S::A_BYTES + S::B_BYTES : S::B_BYTES);
                if constexpr (DENSE) {
                    // the tile's own rows: MT boxes of 128 rows x RB bytes (rows past
                    // the end read as zeros)
#pragma unroll
                    for (int h = 0; h < MT; ++h)
                        ptx::tma_tile2d(a_base + h * kHalf * RB, &tma_a, c0, (int32_t)(row0 + h * kHalf),
                                        &full[s]);
                }
                if constexpr (BMN) {
                    // K = input channels c0.. of offset k (rows of W), N atoms of 64 channels
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        ptx::tma_tile2d(a_base + S::A_BYTES + j * (S::CH * 128), &tma_b, n0 + 64 * j,
                                        k * a.cred + c0, &full[s]);
                } else {
                    ptx::tma_tile2d(a_base + S::A_BYTES, &tma_b, c0, k * a.n_total + n0, &full[s]);
                }
                ++issued;
            }
            // make sure no copy issued above is still landing before the CTA ends
            const int first = issued > STAGES ? issued - STAGES : 0;
            for (int it = first; it < issued; ++it)
                ptx::mbar_wait(&full[it % STAGES], (it / STAGES) & 1, kDrainNs);
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        // B MN-major (the forward's W[k] as stored): transpose bit of the descriptor
        const uint32_t idesc = ptx::idesc_make(TcKind<T>::fmt, kHalf, BN) | (BMN ? 1u << 16 : 0u);
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, a.wait_ns)) {
                atomicExch(&s_ctrl[1], 1);
                break;
            }
            // the rows arrived through generic-proxy copies: order them before
            // the tensor core's async-proxy reads
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_after();
            const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
            // K-major B advances 32 bytes along its rows per instruction; MN-major
            // B advances two 8-row K groups (2048 bytes)
            const uint64_t bd = BMN ? ptx::desc_mn_sw128(a_base + S::A_BYTES, S::CH * 128)
                                    : ptx::desc_k_sw<RB>(a_base + S::A_BYTES);
            constexpr uint64_t kBStep = BMN ? 2048 >> 4 : 2;
#pragma unroll
            for (int kk = 0; kk < RB / 32; ++kk) {  // 32 bytes of K per instruction
                const uint32_t acc = (it | kk) != 0 ? 1u : 0u;
#pragma unroll
                for (int h = 0; h < MT; ++h)
                    ptx::mma<TcKind<T>::kind>(tmem + h * BN,
                                              ptx::desc_k_sw<RB>(a_base + h * kHalf * RB) + 2 * kk,
                                              bd + kBStep * kk, idesc, acc);
            }
            ptx::mma_commit(&empty[s]);
        }
        ptx::mma_commit(done);  // completes once every MMA issued above has finished
    }

    // ---------------------------------------------------------------- epilogue
    if (tid < kWorkers) {
        const bool waited = ptx::mbar_wait(done, 0, kDrainNs);
        ptx::tc_fence_after();
        const bool aborted = __any_sync(FULL_MASK, !waited || s_ctrl[1] != 0);
        // warp w reads TMEM lanes 32*(w%4).. (its lane quarter) of accumulator
        // (w/4)%MT, and column group w/(4 MT) of the tile's BN
        constexpr int kGroups = NW / (4 * MT), kGroupCols = BN / kGroups;
        const int quarter = warp & 3, half = (warp >> 2) % MT, cgrp = warp / (4 * MT);
        const int64_t trow = row0 + half * kHalf + quarter * 32 + lane;
        const bool evalid = trow < a.rows;
        const int64_t erow = evalid && a.perm ? (int64_t)__ldg(a.perm + trow) : trow;
        if (aborted) {
            if (tid == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        } else {
            T* out = static_cast<T*>(a.out);
            const T* bias = static_cast<const T*>(a.bias);
#pragma unroll 1
            constexpr int kCols = kGroupCols >= 32 ? 32 : 16;  // TMEM columns per load
            for (int c = cgrp * kGroupCols; c < (cgrp + 1) * kGroupCols; c += kCols) {
                uint32_t v[kCols];
                if (n_iter > 0) {
                    const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * BN + c);
                    if constexpr (kCols == 32) ptx::tmem_ld32(ta, v);
                    else ptx::tmem_ld16(ta, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < kCols; ++j) v[j] = 0u;
                }
                constexpr int kVec = (int)(kCols * sizeof(T) / 16);  // 16-byte words per chunk
                const bool use_res = a.residual && evalid;
                alignas(16) T rsd[kCols];
                if (use_res) {
                    const uint4* r4 = reinterpret_cast<const uint4*>(
                        static_cast<const T*>(a.residual) + erow * a.n_total + n0 + c);
#pragma unroll
                    for (int q = 0; q < kVec; ++q) reinterpret_cast<uint4*>(rsd)[q] = __ldcs(r4 + q);
                }
                alignas(16) T o[kCols];
#pragma unroll
                for (int j = 0; j < kCols; ++j) {
                    float f = __uint_as_float(v[j]);
                    if (bias) f += elem<T>::to_f32(bias[n0 + c + j]);
                    if (use_res) f = fmaf(a.add_scale, elem<T>::to_f32(rsd[j]), f);
                    if (a.act) f = fmaxf(f, 0.f);
                    o[j] = elem<T>::from_f32(f);
                }
                const uint4* o4 = reinterpret_cast<const uint4*>(o);
                if (S::kTmaStore && tstore) {
                    // into box (half, c / kBoxCols): row r at 128 r, its 16-byte
                    // pieces swizzled by r % 8 as the TMA store reads them
                    constexpr int kBoxCols = 128 / (int)sizeof(T);
                    const int r = quarter * 32 + lane;
                    uint8_t* box = smem + (size_t)(half * (BN / kBoxCols) + c / kBoxCols) * (kHalf * 128);
                    const int j0 = (c % kBoxCols) * (int)sizeof(T) / 16;
#pragma unroll
                    for (int q = 0; q < kVec; ++q)
                        *reinterpret_cast<uint4*>(box + r * 128 + (((j0 + q) ^ (r & 7)) << 4)) = o4[q];
                } else if (evalid) {
                    uint4* d4 = reinterpret_cast<uint4*>(out + erow * a.n_total + n0 + c);
#pragma unroll
                    for (int q = 0; q < kVec; ++q) __stcs(d4 + q, o4[q]);  // streamed out
                }
            }
        }
        if (S::kTmaStore && tstore) {
            // every epilogue thread reaches this barrier (aborted or not); the
            // staged boxes leave once all rows are in place
            if (aborted && lane == 0) atomicExch(&s_ctrl[1], 1);
            ptx::fence_proxy_async_smem();
            ptx::bar_sync_named(1, kWorkers);
            if (tid == 0 && s_ctrl[1] == 0) {
                constexpr int kBoxCols = 128 / (int)sizeof(T);
                for (int h = 0; h < MT; ++h) {
                    const int64_t y = row0 + h * kHalf;
                    if (y >= a.rows) break;  // rows past the end inside a box are clipped
#pragma unroll
                    for (int bx = 0; bx < BN / kBoxCols; ++bx)
                        ptx::tma_store2d(&tma_o, n0 + bx * kBoxCols, (int32_t)y,
                                         ptx::smem_u32(smem + (size_t)(h * (BN / kBoxCols) + bx) * (kHalf * 128)));
                }
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();  // shared memory must outlive the stores' reads
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

// Wt[k][n][c] = W[k][c][n]: the forward's B operand in K-major order.
template <typename T>
__global__ void __launch_bounds__(256) k_transpose_w(const T* __restrict__ w, T* __restrict__ wt,
                                                     int K, int cin, int cout)
{
    __shared__ T tile[32][33];
    const int k = blockIdx.z;
    const int c0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int c = c0 + r, n = n0 + tx;
        if (c < cin && n < cout) tile[r][tx] = w[((int64_t)k * cin + c) * cout + n];
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int n = n0 + r, c = c0 + tx;
        if (c < cin && n < cout) wt[((int64_t)k * cout + n) * cin + c] = tile[tx][r];
    }
}

template <typename T> struct TmaType;
template <> struct TmaType<__half> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; };
template <> struct TmaType<__nv_bfloat16> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; };
template <> struct TmaType<float> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; };

// 2-D row-major [rows, cols] tensor, boxes of RB bytes x box_rows, RB-byte swizzle.
template <typename T, int RB>
bool make_tmap(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    const CUtensorMapSwizzle swz = RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : (RB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    return tmap_2d(m, TmaType<T>::v, (int)sizeof(T), base, cols, rows, (uint32_t)(RB / sizeof(T)),
                   box_rows, swz);
}

template <typename T, int BN, int STAGES, int MT, int NW, int RB, bool BMN, bool DENSE = false>
spc_status launch_tc(const TcArgs& a, cudaStream_t st)
{
    using S = TcShape<T, BN, STAGES, MT, NW, RB>;
    static_assert(NW % (4 * MT) == 0 && (BN / (NW / (4 * MT))) % 16 == 0, "epilogue split");
    static_assert(!BMN || (RB == 128 && sizeof(T) == 2 && BN % 64 == 0), "MN-major B shape");
    CUtensorMap tb;
    // B as stored [K * cred rows][n_total] (boxes of 64 K rows x 64 channels), or
    // transposed [K * n_total rows][cred] (boxes of BN rows x RB bytes)
    const bool tb_ok = BMN ? make_tmap<T, 128>(&tb, a.b, (uint64_t)a.n_total, (uint64_t)a.K * a.cred, S::CH)
                           : make_tmap<T, RB>(&tb, a.b, (uint64_t)a.cred, (uint64_t)a.K * a.n_total, BN);
    if (!tb_ok) return SPC_ERR_UNSUPPORTED;
    // dense A: the input [in_rows][cred] in boxes of 128 rows x RB bytes
    CUtensorMap ta = tb;
    if (DENSE && !make_tmap<T, RB>(&ta, a.in, (uint64_t)a.cred, (uint64_t)a.in_rows, kHalf))
        return SPC_ERR_UNSUPPORTED;
    // Output rows in tile order (no caller permutation) leave through TMA stores
    // when the output is a valid tensor-map target (16-byte aligned base).
    CUtensorMap to = tb;
    int tstore = 0;
    if (S::kTmaStore && a.perm == nullptr) {
        CUtensorMap m;
        if (make_tmap<T, 128>(&m, a.out, (uint64_t)a.n_total, (uint64_t)a.rows, kHalf)) {
            to = m;
            tstore = 1;
        }
    }
    const size_t smem = S::smem_bytes(a.K);
    auto kern = k_conv_tc<T, BN, STAGES, MT, NW, RB, BMN, DENSE>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPC_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S::smem_bytes(32)) != cudaSuccess)
            return SPC_ERR_UNSUPPORTED;
        configured[dev] = true;
    }
    dim3 grid((unsigned)ceil_div(a.rows, S::kRowsPerCta), (unsigned)(a.n_total / BN));
    kern<<<grid, S::kThreads, smem, st>>>(a, tb, to, ta, tstore);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

// Shared memory of one SM (bytes) and what the runtime reserves per CTA.
constexpr size_t kSmemPerSm = 233472, kSmemPerCta = 1024;

template <typename T, int BN, int STAGES, int MT, int NW, int RB>
bool two_per_sm(int K)
{
    return 2 * (TcShape<T, BN, STAGES, MT, NW, RB>::smem_bytes(K) + kSmemPerCta) <= kSmemPerSm;
}

// 128-byte rows: B MN-major (W as stored) when the caller passes it so.
template <typename T, int BN, int STAGES, int MT, int NW>
spc_status launch_wide(const TcArgs& a, cudaStream_t st)
{
    if constexpr (sizeof(T) == 2) {
        if (a.b_mn) return launch_tc<T, BN, STAGES, MT, NW, 128, true>(a, st);
    }
    return launch_tc<T, BN, STAGES, MT, NW, 128, false>(a, st);
}

// K == 1 on the identity map: TMA-loaded row blocks, two CTAs of 2 x 128 rows
// per SM.
template <typename T, int BN>
spc_status launch_dense(const TcArgs& a, cudaStream_t st)
{
    if (a.b_mn) return launch_tc<T, BN, 2, 2, 8, 128, true, true>(a, st);
    return launch_tc<T, BN, 2, 2, 8, 128, false, true>(a, st);
}

template <typename T>
spc_status dispatch_tc(const TcArgs& a, cudaStream_t st)
{
    constexpr int E = (int)sizeof(T);
    if constexpr (E == 2) {
        if (a.map == nullptr && a.K == 1 && a.perm == nullptr && a.cred % 64 == 0 &&
            a.in_rows == a.rows) {
            if (a.n_total % 128 == 0) return launch_dense<T, 128>(a, st);
            if (a.n_total % 64 == 0) return launch_dense<T, 64>(a, st);
        }
    }
    if (a.cred * E % 128 == 0) {
        // Two CTAs per SM wherever the tile's shared memory allows: while one
        // CTA loads its map entries or stores its rows, the other's gathers keep
        // the SM's copy traffic going.  2 x 128-row tiles with 8 gather warps and
        // 2 stages fit when the weight stage is 64 wide (any K up to 31) or when K
        // is small; 128-wide weights with many offsets take 128-row tiles and 3
        // stages.  One CTA of 2 x 128 rows, 16 warps and 4 stages is the shape
        // when neither fits.  Rows in grouped order run only a few offsets per
        // tile and take 128-row tiles.
        if (a.perm && a.n_total % 128 == 0) return launch_wide<T, 128, 2, 1, 8>(a, st);
        if (a.perm) return launch_wide<T, 64, 2, 1, 8>(a, st);
        if (a.n_total % 128 == 0) {
            if (two_per_sm<T, 128, 2, 2, 8, 128>(a.K)) return launch_wide<T, 128, 2, 2, 8>(a, st);
            if (two_per_sm<T, 128, 3, 1, 8, 128>(a.K)) return launch_wide<T, 128, 3, 1, 8>(a, st);
            return launch_wide<T, 128, TC_STAGES, TC_MT, TC_NW>(a, st);
        }
        if (two_per_sm<T, 64, 2, 2, 8, 128>(a.K)) return launch_wide<T, 64, 2, 2, 8>(a, st);
        return launch_wide<T, 64, TC_STAGES, TC_MT, TC_NW>(a, st);
    }
    // narrow rows (32 or 64 bytes): small stages, many CTAs per SM; B K-major
    if (a.b_mn) return SPC_ERR_UNSUPPORTED;
    if (a.cred * E == 64) {
        if (a.n_total == 16) return launch_tc<T, 16, TCN_STAGES, TCN_MT, TCN_NW, 64, false>(a, st);
        if (a.n_total == 32) return launch_tc<T, 32, TCN_STAGES, TCN_MT, TCN_NW, 64, false>(a, st);
        if (a.n_total % 64 == 0) return launch_tc<T, 64, TCN_STAGES, TCN_MT, TCN_NW, 64, false>(a, st);
    } else if (a.cred * E == 32) {
        if (a.n_total == 16) return launch_tc<T, 16, TCN_STAGES, TCN_MT, TCN_NW, 32, false>(a, st);
        if (a.n_total == 32) return launch_tc<T, 32, TCN_STAGES, TCN_MT, TCN_NW, 32, false>(a, st);
        if (a.n_total % 64 == 0) return launch_tc<T, 64, TCN_STAGES, TCN_MT, TCN_NW, 32, false>(a, st);
    }
    return SPC_ERR_UNSUPPORTED;
}

}  // namespace

bool conv_tc_supported(int32_t cred, int32_t cout, int32_t K, spc_dtype dt, spc_precision prec)
{
    if (K < 1 || K > 32) return false;
    const bool wide_n = cout % 64 == 0;
    if (dt == SPC_F16 || dt == SPC_BF16) {
        if (cred % 64 == 0) return wide_n;
        // narrow rows: 16 or 32 channels, N = 16, 32 or a multiple of 64
        return (cred == 16 || cred == 32) && (cout == 16 || cout == 32 || wide_n);
    }
    if (dt == SPC_F32) return prec == SPC_PREC_TF32 && cred % 32 == 0 && wide_n;
    return false;
}

bool conv_tc_reads_w_as_stored(int32_t cin, int32_t cout, spc_dtype dt)
{
    return (dt == SPC_F16 || dt == SPC_BF16) && cin % 64 == 0 && cout % 64 == 0;
}

size_t conv_tc_weight_bytes(int32_t K, int32_t cin, int32_t cout, spc_dtype dt)
{
    return align_up((size_t)K * cin * cout * (dt == SPC_F32 ? 4 : 2), 256);
}

spc_status transpose_weights(const void* w, void* wt, int32_t K, int32_t cin, int32_t cout,
                             spc_dtype dt, cudaStream_t st)
{
    dim3 grid((unsigned)ceil_div(cout, 32), (unsigned)ceil_div(cin, 32), (unsigned)K);
    switch (dt) {
    case SPC_F32:
        k_transpose_w<float><<<grid, 256, 0, st>>>(static_cast<const float*>(w),
                                                   static_cast<float*>(wt), K, cin, cout);
        break;
    case SPC_F16:
        k_transpose_w<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(w),
                                                    static_cast<__half*>(wt), K, cin, cout);
        break;
    case SPC_BF16:
        k_transpose_w<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(wt), K, cin, cout);
        break;
    }
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

spc_status conv_gather_tc(const TcArgs& a, spc_dtype dt, cudaStream_t st)
{
    if (a.rows == 0) return SPC_OK;
    switch (dt) {
    case SPC_F16: return dispatch_tc<__half>(a, st);
    case SPC_BF16: return dispatch_tc<__nv_bfloat16>(a, st);
    case SPC_F32: return dispatch_tc<float>(a, st);
    }
    return SPC_ERR_INVALID_ARG;
}

}  // namespace spc
