// conv_i8.cu -- quantized (int8) gathered implicit GEMM on the tcgen05 tensor
// cores, with spconv's per-output-channel scale and bias, fused residual add
// and ReLU, and a saturating int8 output (spconv docs, TENSORRT_INT8_GUIDE.md:
// "Spconv Int8 Scale/Bias Conversion Basic Rule", "Call Spconv Implicit GEMM
// with Calculated Scales and Bias").
//
// sm_103a has no integer MMA (ptxas rejects tcgen05.mma .kind::i8 for this
// target), so the integer sums are formed exactly on the fp16 path.  Every
// int8 value is exact in fp16 (|v| <= 128 < 2^11), every product of two is an
// exact fp32 integer (|x w| <= 2^14), and a sum of integers stays exact in fp32
// while every partial sum is below 2^24 in magnitude, whatever the order.  Two
// ways keep the partial sums in range:
//   * several accumulators (NACC > 0): stage t (64 input channels of one
//     offset) accumulates into tensor-memory accumulator t % NACC, so an
//     accumulator sums at most 15 stages (960 products, |sum| < 2^24), and the
//     epilogue adds the NACC accumulators in int32.  The weights are only
//     widened to fp16 (a K-major B operand of BN rows per CTA); the MMA is
//     N = BN wide.  Needs K * Cin / 64 <= 15 NACC with NACC * BN <= 512 TMEM
//     columns (K * Cin <= 7680);
//   * a 4-bit weight split (NACC = 0, up to K * Cin = 8192): w = 16 * hi + lo,
//     hi in [-8, 7], lo in [0, 15], prepared once per call as a K-major B
//     operand of 2 * BN rows per CTA (the hi rows, then the lo rows); one MMA
//     of N = 2 * BN accumulates sum x * hi and sum x * lo side by side
//     (|x * lo| <= 1920, so 8192 products stay below 2^24), and the epilogue
//     forms acc = 16 * hi_sum + lo_sum in int32.
// The epilogue then computes f = float(acc) * scale + bias (+ add_scale *
// float(add)), ReLU, rounds half away from zero and saturates to [-128, 127],
// each fp32 operation rounded once in that order.
//
// The gather stays on int8 rows (half the bytes of a 16-bit row): gather warps
// copy each tile row's 64-byte int8 chunk with 16-byte cp.async into a raw
// ring in shared memory (a thread later reads only the pieces it copied
// itself, so the ring needs no barrier), widen them to fp16 in registers, and
// write them to the 128-byte-swizzled K-major stage the MMA reads; the stage's
// mbarrier completes when every gather thread has written its pieces and the
// weight tile's TMA has landed.  Tiles, map prologue, row order (`perm`, the
// do_sort variant; NULL keeps rows in map order), bounded waits and the
// single-writer output match the 16-bit kernel (conv_tc.cu).
#include "conv_tile.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace spc {

namespace {

constexpr int kRows = 128;  // output rows per CTA (one MMA of M = 128)
constexpr int kCh = 64;     // input channels per stage (128 bytes of fp16)
constexpr uint64_t kDrainNs = 2000000000ull;  // bound of the waits for a CTA's own copies / MMAs

template <int BN, int STAGES, int NW, int RAW, int NACC>
struct I8Shape {
    static constexpr int kWorkers = NW * 32;
    static constexpr int kThreads = kWorkers + 64;
    static constexpr int kTmaWarp = NW, kMmaWarp = NW + 1;
    static constexpr int A_BYTES = kRows * 128;         // 128 rows x 64 fp16
    static constexpr int BROWS = NACC ? BN : 2 * BN;    // B rows: the weights, or their hi and lo halves
    static constexpr int B_BYTES = BROWS * 128;         // x 64 fp16
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int RAW_BYTES = kRows * kCh;       // 128 rows x 64 int8
    static constexpr int PIECES = kRows * kCh / 16;     // 16-byte pieces per stage
    static constexpr int PER_THREAD = PIECES / kWorkers;
    static constexpr int ACC_COLS = NACC ? NACC * BN : 2 * BN;
    static constexpr int TMEM_COLS = ACC_COLS <= 128 ? 128 : (ACC_COLS <= 256 ? 256 : 512);
    static constexpr int kMinCtas = TMEM_COLS <= 128 && STAGES <= 2 ? 2 : 1;
    static_assert(ACC_COLS <= 512, "tensor memory");
    static_assert(PIECES % kWorkers == 0, "pieces per thread");
    static size_t smem_bytes(int K)
    {
        return 1024 + (size_t)STAGES * STAGE_BYTES + (size_t)RAW * RAW_BYTES + (size_t)K * kRows * 4 +
               8 * (2 * STAGES + 1) + 4 * 40;
    }
};

// Four int8 values (one 32-bit word) to four exact fp16 values (two words):
// with u = v + 128 (the byte with its top bit flipped), the fp16 bit pattern
// 0x6400 | u is 1024 + u (binary16: exponent 25, u in the low mantissa bits),
// and subtracting 1152 = 1024 + 128 leaves v exactly.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // bytes u0, 0x64, u1, 0x64
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // bytes u2, 0x64, u3, 0x64
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480),
                                        __ushort_as_half((unsigned short)0x6480));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

template <int BN, int STAGES, int NW, int RAW, int NACC>
__global__ void __launch_bounds__(I8Shape<BN, STAGES, NW, RAW, NACC>::kThreads, I8Shape<BN, STAGES, NW, RAW, NACC>::kMinCtas)
k_conv_i8(I8Args a, const __grid_constant__ CUtensorMap tma_b)
{
    using S = I8Shape<BN, STAGES, NW, RAW, NACC>;
    constexpr int kWorkers = S::kWorkers, kTmaWarp = S::kTmaWarp, kMmaWarp = S::kMmaWarp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw = smem + (size_t)STAGES * S::STAGE_BYTES;
    int32_t* s_idx = reinterpret_cast<int32_t*>(raw + (size_t)RAW * S::RAW_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(s_idx + (size_t)a.K * kRows);
    uint64_t* empty = full + STAGES;
    uint64_t* done = empty + STAGES;
    int* s_active = reinterpret_cast<int*>(done + 1);  // [32]
    int* s_ctrl = s_active + 32;                      // nact, abort, union, tmem
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kRows;
    const int blk = blockIdx.y, n0 = blk * BN;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], kWorkers + 1);  // every gather thread + the weight TMA
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        s_ctrl[0] = 0;
        s_ctrl[1] = 0;
        s_ctrl[2] = 0;
        ptx::mbar_init_fence();
    }
    if (warp == kTmaWarp && lane == 0) ptx::prefetch_tmap(&tma_b);
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&s_ctrl[3]), S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const TileMap tm{a.map, a.mask, a.perm, a.rows, a.in_rows, a.K, 0};
    const int nact = tile_map_entries<kRows>(tm, row0, tid, s_idx, s_active, &s_ctrl[0],
                                             reinterpret_cast<unsigned*>(&s_ctrl[2]));
    const int kchunks = a.cin / kCh;
    const int n_iter = nact * kchunks;
    const uint32_t tmem = (uint32_t)s_ctrl[3];

    if (tid < kWorkers) {
        // ------------------------------------------- int8 row gathers + widening
        // piece e = j * kWorkers + tid: tile row e / 4, 16 input channels
        // 16 (e % 4) .. of the stage's 64; each becomes two 16-byte fp16 pieces
        // of the row's 128-byte swizzled line.
        const int8_t* in = a.in;
        const uint64_t keep = ptx::policy_evict_last();
        const uint32_t raw_base = ptx::smem_u32(raw);
        auto issue = [&](int q) {
            const int ai = q / kchunks;
            const int c0 = (q % kchunks) * kCh;
            const int32_t* idx = s_idx + ai * kRows;
            const uint32_t slot = raw_base + (uint32_t)((q % RAW) * S::RAW_BYTES);
#pragma unroll
            for (int j = 0; j < S::PER_THREAD; ++j) {
                const int e = j * kWorkers + tid;
                const int r = e >> 2, p = e & 3;
                const int32_t i = idx[r];
                const int8_t* src = i >= 0 ? in + (int64_t)i * a.cin + c0 + p * 16 : in;
                ptx::cp_async16_hint(slot + (uint32_t)(r * kCh + p * 16), src, i >= 0 ? 16u : 0u, keep);
            }
        };
#pragma unroll
        for (int q = 0; q < RAW; ++q) {
            if (q < n_iter) issue(q);
            ptx::cp_async_commit();
        }
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            ptx::cp_async_wait<RAW - 1>();  // this thread's copies of iteration `it` have landed
            if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, a.wait_ns)) {
                atomicExch(&s_ctrl[1], 1);
                break;
            }
            const uint8_t* slot = raw + (size_t)(it % RAW) * S::RAW_BYTES;
            uint8_t* stage = smem + (size_t)s * S::STAGE_BYTES;
#pragma unroll
            for (int j = 0; j < S::PER_THREAD; ++j) {
                const int e = j * kWorkers + tid;
                const int r = e >> 2, p = e & 3;
                const uint4 v = *reinterpret_cast<const uint4*>(slot + r * kCh + p * 16);
                uint4 o0, o1;
                i8x4_to_f16x4(v.x, o0.x, o0.y);
                i8x4_to_f16x4(v.y, o0.z, o0.w);
                i8x4_to_f16x4(v.z, o1.x, o1.y);
                i8x4_to_f16x4(v.w, o1.z, o1.w);
                const int sw = r & 7;
                *reinterpret_cast<uint4*>(stage + r * 128 + (((2 * p) ^ sw) << 4)) = o0;
                *reinterpret_cast<uint4*>(stage + r * 128 + (((2 * p + 1) ^ sw) << 4)) = o1;
            }
            // the fp16 rows were written through the generic proxy: order them
            // before the tensor core's async-proxy reads, then signal the stage
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&full[s]);
            if (it + RAW < n_iter) issue(it + RAW);
            ptx::cp_async_commit();
        }
        ptx::cp_async_wait_all();  // nothing of ours may still land when the CTA ends
    } else if (warp == kTmaWarp) {
        // ---------------------------------- fp16 weights or halves (TMA, K-major)
        int issued = 0;
        if (lane == 0) {
            const int nblk = a.cout / BN;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it % STAGES;
                if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, a.wait_ns)) {
                    atomicExch(&s_ctrl[1], 1);
                    break;
                }
                const int k = s_active[it / kchunks];
                const int c0 = (it % kchunks) * kCh;
                const uint32_t b_dst = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES + S::A_BYTES);
                ptx::mbar_arrive_expect_tx(&full[s], S::B_BYTES);
                ptx::tma_tile2d(b_dst, &tma_b, c0, (k * nblk + blk) * S::BROWS, &full[s]);
                ++issued;
            }
            const int first = issued > STAGES ? issued - STAGES : 0;
            for (int it = first; it < issued; ++it)
                ptx::mbar_wait(&full[it % STAGES], (it / STAGES) & 1, kDrainNs);
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        const uint32_t idesc = ptx::idesc_make(0 /* fp16 */, kRows, S::BROWS);
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, a.wait_ns)) {
                atomicExch(&s_ctrl[1], 1);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
            const uint64_t ad = ptx::desc_k_sw<128>(a_base);
            const uint64_t bd = ptx::desc_k_sw<128>(a_base + S::A_BYTES);
            // several accumulators: stage it goes to accumulator it % NACC, whose
            // first stage overwrites it
            const uint32_t d = NACC ? tmem + (uint32_t)((it % (NACC ? NACC : 1)) * BN) : tmem;
            const bool first = NACC ? it < NACC : it == 0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 channels (32 bytes) of K per instruction
                ptx::mma<0>(d, ad + 2 * kk, bd + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
            ptx::mma_commit(&empty[s]);
        }
        ptx::mma_commit(done);
    }

    // ---------------------------------------------------------------- epilogue
    if (tid < kWorkers) {
        const bool waited = ptx::mbar_wait(done, 0, kDrainNs);
        ptx::tc_fence_after();
        const bool aborted = __any_sync(FULL_MASK, !waited || s_ctrl[1] != 0);
        // warp w reads TMEM lanes 32 (w % 4).. and column group w / 4 of BN
        constexpr int kGroups = NW / 4, kGroupCols = BN / kGroups;
        const int quarter = warp & 3, cgrp = warp >> 2;
        const int64_t trow = row0 + quarter * 32 + lane;
        const bool evalid = trow < a.rows;
        const int64_t erow = evalid && a.perm ? (int64_t)__ldg(a.perm + trow) : trow;
        if (aborted) {
            if (tid == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        } else {
#pragma unroll 1
            for (int c = cgrp * kGroupCols; c < (cgrp + 1) * kGroupCols; c += 16) {
                int acc[16];
                if (NACC) {
                    // the sum of the accumulators that received stages (exact integers)
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0;
                    const int na = n_iter < NACC ? n_iter : NACC;
                    for (int q = 0; q < na; ++q) {
                        uint32_t v[16];
                        ptx::tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(q * BN + c), v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] += __float2int_rn(__uint_as_float(v[j]));
                    }
                } else {
                    uint32_t vh[16], vl[16];
                    if (n_iter > 0) {
                        const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16);
                        ptx::tmem_ld16(ta + (uint32_t)c, vh);
                        ptx::tmem_ld16(ta + (uint32_t)(BN + c), vl);
                        ptx::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) vh[j] = vl[j] = 0u;
                    }
                    // exact integers: |hi sum| < 2^23, 0 <= |lo sum| < 2^24
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        acc[j] = __float2int_rn(__uint_as_float(vh[j])) * 16 + __float2int_rn(__uint_as_float(vl[j]));
                }
                const int n = n0 + c;
                alignas(16) int8_t add[16];
                const bool use_add = a.add && evalid;
                if (use_add)
                    *reinterpret_cast<uint4*>(add) =
                        __ldcs(reinterpret_cast<const uint4*>(a.add + erow * a.cout + n));
                alignas(16) int8_t o[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float f = __fmul_rn(__int2float_rn(acc[j]), __ldg(a.scale + n + j));
                    if (a.bias) f = __fadd_rn(f, __ldg(a.bias + n + j));
                    if (use_add) f = __fadd_rn(f, __fmul_rn(a.add_scale, (float)add[j]));
                    if (a.act && f < 0.f) f = 0.f;
                    f = fminf(fmaxf(roundf(f), -128.f), 127.f);
                    o[j] = (int8_t)(int)f;
                }
                if (evalid) __stcs(reinterpret_cast<uint4*>(a.out + erow * a.cout + n), *reinterpret_cast<const uint4*>(o));
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

// wq[k][blk][r][c] (fp16, [K][cout / BN][rows][cin]).  split: rows = 2 BN, for
// r < BN the high part of w[k][c][blk BN + r], else the low part of
// w[k][c][blk BN + r - BN], with w = 16 hi + lo, hi = floor(w / 16) in [-8, 7],
// lo in [0, 15].  Otherwise rows = BN and the weight itself.
__global__ void k_i8_prep_w(const int8_t* __restrict__ w, __half* __restrict__ wq, int K, int cin,
                            int cout, int bn, int split)
{
    const int rows = split ? 2 * bn : bn;
    const int64_t total = (int64_t)K * (cout / bn) * rows * cin;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % cin);
        int64_t t = e / cin;
        const int r = (int)(t % rows);
        t /= rows;
        const int blk = (int)(t % (cout / bn));
        const int k = (int)(t / (cout / bn));
        const int ch = blk * bn + (r < bn ? r : r - bn);
        const int v = w[((int64_t)k * cin + c) * cout + ch];
        const int part = !split ? v : (r < bn ? (v >> 4) : (v & 15));
        wq[e] = __int2half_rn(part);
    }
}

constexpr size_t kSmemPerSm = 233472, kSmemPerCta = 1024;

template <int BN, int STAGES, int NW, int RAW, int NACC>
spc_status launch_i8(const I8Args& a, const int8_t* w, cudaStream_t st)
{
    using S = I8Shape<BN, STAGES, NW, RAW, NACC>;
    const int64_t total = (int64_t)a.K * (a.cout / BN) * S::BROWS * a.cin;
    const int blocks = (int)std::min<int64_t>(ceil_div(total, 256), 4096);
    k_i8_prep_w<<<blocks, 256, 0, st>>>(w, a.wq, a.K, a.cin, a.cout, BN, NACC ? 0 : 1);
    SPC_LAUNCH_CHECK();
    CUtensorMap tb;
    if (!tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.wq, (uint64_t)a.cin,
                 (uint64_t)a.K * (a.cout / BN) * S::BROWS, kCh, S::BROWS, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPC_ERR_UNSUPPORTED;
    const size_t smem = S::smem_bytes(a.K);
    auto kern = k_conv_i8<BN, STAGES, NW, RAW, NACC>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPC_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S::smem_bytes(32)) != cudaSuccess)
            return SPC_ERR_UNSUPPORTED;
        configured[dev] = true;
    }
    dim3 grid((unsigned)ceil_div(a.rows, kRows), (unsigned)(a.cout / BN));
    kern<<<grid, S::kThreads, smem, st>>>(a, tb);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

}  // namespace

bool conv_i8_supported(int32_t K, int32_t cin, int32_t cout)
{
    // K * cin <= 8192 keeps every fp32 partial sum an exact integer
    return K >= 1 && K <= 32 && cin % 64 == 0 && cout % 64 == 0 && (int64_t)K * cin <= 8192;
}

size_t conv_i8_ws_bytes(int32_t K, int32_t cin, int32_t cout)
{
    // the larger of the two weight layouts (the split one)
    return align_up((size_t)K * 2 * cout * cin * sizeof(__half), 256);
}

spc_status conv_i8(const I8Args& a, const int8_t* w, cudaStream_t st)
{
    if (a.rows == 0) return SPC_OK;
    // accumulators needed so that none sums more than 15 stages of 64 channels
    const int64_t stages = (int64_t)a.K * (a.cin / kCh);
    const int64_t nacc = ceil_div(stages, 15);
    if (a.cout % 128 == 0 && nacc <= 4) return launch_i8<128, 4, 8, 4, 4>(a, w, st);
    if (nacc <= 8) return launch_i8<64, 4, 8, 4, 8>(a, w, st);
    if (a.cout % 128 == 0) return launch_i8<128, 3, 8, 4, 0>(a, w, st);
    return launch_i8<64, 2, 8, 3, 0>(a, w, st);
}

}  // namespace spc
