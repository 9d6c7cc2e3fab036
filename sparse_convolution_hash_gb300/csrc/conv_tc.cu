// conv_tc.cu -- gathered implicit GEMM on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory) for wide channels.
//
// Output-stationary: a CTA owns 128 output rows (the MMA's M) x BN output
// channels.  It first ORs its rows' offset masks, so offsets that no row of
// the tile uses are skipped, and reads its rows' map entries for the remaining
// offsets.  The K loop then runs over (active offset, 128-byte channel chunk):
//   producers (warps 0-3, one row each) gather the 128 input rows of that
//     offset with 16-byte cp.async copies straight into a 128-byte-swizzled
//     K-major shared-memory stage (rows with no neighbour are zero-filled by
//     the copy itself), plus the matching BN x 128-byte weight tile;
//   one thread of warp 4 waits for the stage, issues four tcgen05.mma (K = 32
//     bytes each) into the fp32 accumulator in tensor memory, and commits the
//     stage back to the producers.
// All offsets accumulate in tensor memory; the epilogue (warps 0-3) reads each
// row's accumulators with tcgen05.ld, adds the bias, rounds once and stores the
// row.  Every output row is written once: no atomics, run-to-run identical.
//
// Forward: B = the weight slice transposed to [Cout][Cin] (K-major), prepared
// once per call in the workspace.  dinput: rows are input rows, the map is the
// transposed or mirrored map, and B = W[k] as stored ([Cin][Cout] is already
// [N][K] K-major for that product).
//
// Every barrier wait is bounded (2 s of wall time); a wait that runs out sets
// SPC_ERR_TIMEOUT in the status word, the CTA drains its copies, waits for its
// MMAs, frees its tensor memory and returns.
#include "kernels.cuh"
#include "ptx.cuh"

namespace spc {

namespace {

constexpr int kRowsPerCta = 128;
constexpr int kThreads = 160;
constexpr uint64_t kWaitNs = 2000000000ull;

template <typename T, int BN, int STAGES>
struct TcShape {
    static constexpr int ELEM = (int)sizeof(T);
    static constexpr int CH = 128 / ELEM;  // elements per 128-byte chunk of a row
    static constexpr int A_BYTES = kRowsPerCta * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
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

template <typename T, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) k_conv_tc(TcArgs a)
{
    using S = TcShape<T, BN, STAGES>;
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
    const uint32_t kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], kRowsPerCta);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        s_ctrl[0] = 0;
        s_ctrl[1] = 0;
        s_ctrl[2] = 0;
        ptx::mbar_init_fence();
    }
    if (warp == 4) {
        ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&s_ctrl[3]), BN);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // union of the tile's row masks
    const int64_t row = row0 + tid;
    const bool rvalid = tid < kRowsPerCta && row < a.rows;
    uint32_t m = 0;
    if (tid < kRowsPerCta) {
        if (rvalid) {
            m = a.mask ? a.mask[row] : kmask;
            if (a.mask && a.mirror) m = __brev(m) >> (32 - K);
            m &= kmask;
        }
        const uint32_t wu = __reduce_or_sync(FULL_MASK, m);
        if (lane == 0 && wu) atomicOr(reinterpret_cast<unsigned*>(&s_ctrl[2]), wu);
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t u = (uint32_t)s_ctrl[2];
        int n = 0;
        while (u) {
            s_active[n++] = __ffs(u) - 1;
            u &= u - 1;
        }
        s_ctrl[0] = n;
    }
    __syncthreads();
    const int nact = s_ctrl[0];
    const int kchunks = a.cred / S::CH;
    const int n_iter = nact * kchunks;
    const uint32_t tmem = (uint32_t)s_ctrl[3];
    const uint8_t* in = static_cast<const uint8_t*>(a.in);
    const uint8_t* bmat = static_cast<const uint8_t*>(a.b);

    if (tid < kRowsPerCta) {
        // ---------------------------------------------------------- producers
        for (int ai = 0; ai < nact; ++ai) {
            const int k = s_active[ai];
            int32_t i = -1;
            if (rvalid && ((m >> k) & 1u)) {
                const int mk = a.mirror ? K - 1 - k : k;
                i = a.map ? a.map[(int64_t)mk * a.rows + row] : (int32_t)row;
                if (i >= a.in_rows) i = -1;
            }
            s_idx[ai * kRowsPerCta + tid] = i;
        }
        bool ok = true;
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            if (it >= STAGES && !ptx::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, kWaitNs)) {
                ok = false;
                break;
            }
            const int ai = it / kchunks;
            const int c0 = (it % kchunks) * S::CH;
            const int k = s_active[ai];
            const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
            const uint32_t b_base = a_base + S::A_BYTES;
            const int32_t i = s_idx[ai * kRowsPerCta + tid];
            const uint8_t* src = i >= 0 ? in + ((int64_t)i * a.cred + c0) * S::ELEM : in;
            const uint32_t nbytes = i >= 0 ? 16u : 0u;
            const uint32_t arow = a_base + (uint32_t)tid * 128u;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                ptx::cp_async16(arow + ((uint32_t)(ch ^ (tid & 7)) << 4), src + (i >= 0 ? ch * 16 : 0),
                                nbytes);
            const uint8_t* bk = bmat + (((int64_t)k * a.n_total + n0) * a.cred + c0) * S::ELEM;
#pragma unroll
            for (int e = tid; e < BN * 8; e += kRowsPerCta) {
                const int r = e >> 3, ch = e & 7;
                ptx::cp_async16(b_base + (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4),
                                bk + (int64_t)r * a.cred * S::ELEM + ch * 16, 16u);
            }
            ptx::cp_async_commit();
            if (it >= STAGES - 1) {
                ptx::cp_async_wait<STAGES - 1>();
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&full[(it - (STAGES - 1)) % STAGES]);
            }
        }
        ptx::cp_async_wait_all();
        ptx::fence_proxy_async_smem();
        if (ok) {
            for (int j = n_iter - (STAGES - 1) > 0 ? n_iter - (STAGES - 1) : 0; j < n_iter; ++j)
                ptx::mbar_arrive(&full[j % STAGES]);
        } else {
            atomicExch(&s_ctrl[1], 1);
        }
    } else if (warp == 4 && lane == 0) {
        // ------------------------------------------------------- MMA issuer
        const uint32_t idesc = ptx::idesc_make(TcKind<T>::fmt, kRowsPerCta, BN);
        for (int it = 0; it < n_iter; ++it) {
            const int s = it % STAGES;
            if (!ptx::mbar_wait(&full[s], (it / STAGES) & 1, kWaitNs)) {
                atomicExch(&s_ctrl[1], 1);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * S::STAGE_BYTES);
            const uint64_t ad = ptx::desc_k_sw128(a_base);
            const uint64_t bd = ptx::desc_k_sw128(a_base + S::A_BYTES);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 32 bytes of K per instruction
                ptx::mma<TcKind<T>::kind>(tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                          (it | kk) != 0 ? 1u : 0u);
            ptx::mma_commit(&empty[s]);
        }
        ptx::mma_commit(done);  // completes once every MMA issued above has finished
    }

    // ---------------------------------------------------------------- epilogue
    if (tid < kRowsPerCta) {
        const bool waited = ptx::mbar_wait(done, 0, kWaitNs);
        ptx::tc_fence_after();
        const bool aborted = __any_sync(FULL_MASK, !waited || s_ctrl[1] != 0);
        if (aborted) {
            if (tid == 0) set_status(a.status, SPC_ERR_TIMEOUT);
        } else {
            T* out = static_cast<T*>(a.out);
            const T* bias = static_cast<const T*>(a.bias);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                if (n_iter > 0) {
                    ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
                if (rvalid) {
                    T* dst = out + row * a.n_total + n0 + c;
                    alignas(16) T o[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float f = __uint_as_float(v[j]);
                        if (bias) f += elem<T>::to_f32(bias[n0 + c + j]);
                        o[j] = elem<T>::from_f32(f);
                    }
                    const uint4* o4 = reinterpret_cast<const uint4*>(o);
                    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int q = 0; q < (int)(32 * sizeof(T) / 16); ++q) d4[q] = o4[q];
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, BN);
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

template <typename T, int BN, int STAGES>
spc_status launch_tc(const TcArgs& a, cudaStream_t st)
{
    using S = TcShape<T, BN, STAGES>;
    const size_t smem = S::smem_bytes(a.K);
    auto kern = k_conv_tc<T, BN, STAGES>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPC_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S::smem_bytes(32)) != cudaSuccess)
            return SPC_ERR_UNSUPPORTED;
        configured[dev] = true;
    }
    dim3 grid((unsigned)ceil_div(a.rows, kRowsPerCta), (unsigned)(a.n_total / BN));
    kern<<<grid, kThreads, smem, st>>>(a);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

template <typename T>
spc_status dispatch_tc(const TcArgs& a, cudaStream_t st)
{
    // stage counts keep two CTAs' shared memory on one SM
    if (a.n_total % 128 == 0) return launch_tc<T, 128, 3>(a, st);
    return launch_tc<T, 64, 4>(a, st);
}

}  // namespace

bool conv_tc_supported(int32_t cred, int32_t cout, int32_t K, spc_dtype dt, spc_precision prec)
{
    if (K < 1 || K > 32 || cout % 64 != 0) return false;
    if (dt == SPC_F16 || dt == SPC_BF16) return cred % 64 == 0;
    if (dt == SPC_F32) return prec == SPC_PREC_TF32 && cred % 32 == 0;
    return false;
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
