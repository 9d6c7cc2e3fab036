// conv_narrow.cu -- gathered conv for narrow channels (Cin, Cout in {8, 16, 32}).
//
// Narrow layers move far more bytes than they compute (a 16 -> 16 pair is 256
// multiply-adds on a 32-byte row), and on sparse scenes most rows have only a
// few neighbours, so this path is laid out for latency, not for tensor cores:
// one thread owns one output row and keeps its Cout fp32 accumulators in
// registers; the weight tensor is converted to fp32 once per persistent block
// and kept in shared memory (each offset's slice padded by 16 bytes, so lanes
// reading different offsets' slices spread over the banks).  A thread walks
// only its own row's offset mask, a few offsets at a time: their map entries
// are loaded together, then their neighbours' rows (16-byte vector loads),
// then the multiply-adds run.  A row with at most that many neighbours costs
// two dependent memory round trips.  Rows are written once, with vector
// stores.  Blocks are sized so that the whole grid is resident at once.
//
// The same kernel computes dinput with the transposed weight slice and the
// transposed map (or the submanifold map read through its offset mirror, in
// which case the mask bits are mirrored too).
#include "kernels.cuh"

namespace spc {

namespace {

constexpr int kThreads = 256;

template <typename T, int N>
struct RowVec {
    // N elements of T moved as 16-byte words
    static constexpr int kWords = (N * (int)sizeof(T)) / 16;
    uint4 w[kWords];
};

template <typename T, int CRED, int COUT>
__device__ __forceinline__ void fma_row(float (&acc)[COUT], const RowVec<T, CRED>& xv,
                                        const float* __restrict__ wk)
{
    const T* xe = reinterpret_cast<const T*>(xv.w);
    const float4* w4 = reinterpret_cast<const float4*>(wk);
#pragma unroll 4
    for (int c = 0; c < CRED; ++c) {
        const float xc = elem<T>::to_f32(xe[c]);
#pragma unroll
        for (int j4 = 0; j4 < COUT / 4; ++j4) {
            const float4 wv = w4[c * (COUT / 4) + j4];
            acc[4 * j4 + 0] = fmaf(xc, wv.x, acc[4 * j4 + 0]);
            acc[4 * j4 + 1] = fmaf(xc, wv.y, acc[4 * j4 + 1]);
            acc[4 * j4 + 2] = fmaf(xc, wv.z, acc[4 * j4 + 2]);
            acc[4 * j4 + 3] = fmaf(xc, wv.w, acc[4 * j4 + 3]);
        }
    }
}

template <typename T, int N>
__device__ __forceinline__ void load_row(RowVec<T, N>& v, const T* __restrict__ base, int32_t i)
{
    const uint4* src = reinterpret_cast<const uint4*>(base + (int64_t)i * N);
#pragma unroll
    for (int q = 0; q < RowVec<T, N>::kWords; ++q) v.w[q] = __ldg(src + q);
}

// fp32 words between consecutive offsets' weight slices in shared memory
template <int CRED, int COUT>
constexpr int kSliceStride = CRED * COUT + 4;

template <typename T, int CRED, int COUT>
constexpr int kNarrowBatch = CRED * (int)sizeof(T) >= 64 ? 1 : (CRED * (int)sizeof(T) >= 32 ? 2 : 4);

// Up to kBatch of the offsets left in m (lowest first, removed from m) and
// their map entries (loads in flight together).
template <int kBatch>
__device__ __forceinline__ void take_batch(uint32_t& m, const GatherGemm& p, int64_t r, int (&ks)[kBatch],
                                           int32_t (&idx)[kBatch])
{
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
        ks[b] = m ? __ffs(m) - 1 : -1;
        m &= m - 1;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
        idx[b] = -1;
        if (ks[b] >= 0) {
            const int mk = p.mirror ? p.K - 1 - ks[b] : ks[b];
            idx[b] = p.map ? __ldcs(p.map + (int64_t)mk * p.rows + r) : (int32_t)r;
        }
    }
}

// The neighbour rows of a batch (loads in flight together).
template <typename T, int CRED, int kBatch>
__device__ __forceinline__ void load_rows(const GatherGemm& p, const int32_t (&idx)[kBatch],
                                          RowVec<T, CRED> (&xv)[kBatch])
{
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
        if (idx[b] >= 0) load_row(xv[b], static_cast<const T*>(p.in), idx[b]);
}

template <typename T, int CRED, int COUT>
__global__ void __launch_bounds__(kThreads, (COUT <= 16 ? 4 : 2)) k_conv_narrow(GatherGemm p)
{
    // offsets whose map entries and rows are in flight together
    constexpr int kBatch = kNarrowBatch<T, CRED, COUT>;
    constexpr int kStr = kSliceStride<CRED, COUT>;
    extern __shared__ __align__(16) float s_w[];  // [K][kStr] fp32 ([CRED][COUT] + pad), then bias [COUT]
    const T* __restrict__ in = static_cast<const T*>(p.in);
    const int K = p.K;
    const uint32_t kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;

    // The first row's mask, map entries and neighbour rows are requested before
    // the block stages its weights, so the two latencies overlap.
    uint32_t m = 0;
    int ks[kBatch];
    int32_t idx[kBatch];
    RowVec<T, CRED> xv[kBatch];
    bool have_rows = false;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) idx[b] = -1;
    if (p.mask && r < p.rows) {
        m = __ldcs(p.mask + r);  // read once: evict first
        if (p.mirror) m = __brev(m) >> (32 - K);
        m &= kmask;
        take_batch<kBatch>(m, p, r, ks, idx);
        load_rows<T, CRED, kBatch>(p, idx, xv);
        have_rows = true;
    }
    {
        // weights: 16-byte vector loads in global order, converted to fp32
        constexpr int kPer = 16 / (int)sizeof(T);
        const int total = K * CRED * COUT;
        const uint4* w4 = static_cast<const uint4*>(p.w);
        for (int v0 = threadIdx.x; v0 * kPer < total; v0 += blockDim.x * 4) {
            uint4 buf[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v * kPer < total) buf[u] = __ldg(w4 + v);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v * kPer >= total) continue;
                const T* e = reinterpret_cast<const T*>(&buf[u]);
#pragma unroll
                for (int t = 0; t < kPer; ++t) {
                    const int g = v * kPer + t;  // global element index
                    const int k = g / (CRED * COUT);
                    int a = (g / COUT) % CRED, b = g % COUT;  // [K][CRED][COUT] order
                    if (p.transpose_w) {  // global [K][COUT][CRED]
                        a = g % CRED;
                        b = (g / CRED) % COUT;
                    }
                    s_w[k * kStr + a * COUT + b] = elem<T>::to_f32(e[t]);
                }
            }
        }
    }
    float* s_bias = s_w + (size_t)K * kStr;
    for (int j = threadIdx.x; j < COUT; j += blockDim.x)
        s_bias[j] = p.bias ? elem<T>::to_f32(static_cast<const T*>(p.bias)[j]) : 0.f;
    __syncthreads();

    for (bool first = true; r < p.rows; r += step, first = false) {
        float acc[COUT];
#pragma unroll
        for (int j = 0; j < COUT; ++j) acc[j] = s_bias[j];

        if (p.mask) {
            if (!first) {
                m = __ldcs(p.mask + r);
                if (p.mirror) m = __brev(m) >> (32 - K);
                m &= kmask;
                take_batch<kBatch>(m, p, r, ks, idx);
                have_rows = false;
            }
            // the next batch's map entries are requested while this batch's rows
            // load, so a row of n batches costs about n + 1 round trips, not 2n
            while (true) {
                int ks2[kBatch];
                int32_t idx2[kBatch];
                const bool more = m != 0;
                if (more) take_batch<kBatch>(m, p, r, ks2, idx2);
                if (!have_rows) load_rows<T, CRED, kBatch>(p, idx, xv);
                have_rows = false;
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (idx[b] >= 0) fma_row<T, CRED, COUT>(acc, xv[b], s_w + (size_t)ks[b] * kStr);
                if (!more) break;
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    ks[b] = ks2[b];
                    idx[b] = idx2[b];
                }
            }
        } else {
            for (int k = 0; k < K; ++k) {
                const int mk = p.mirror ? K - 1 - k : k;
                const int32_t i = p.map ? p.map[(int64_t)mk * p.rows + r] : (int32_t)r;
                if (i < 0) continue;
                RowVec<T, CRED> xr;
                load_row(xr, in, i);
                fma_row<T, CRED, COUT>(acc, xr, s_w + (size_t)k * kStr);
            }
        }
        if (p.residual) {  // fused residual add, before the activation
            RowVec<T, COUT> rv;
            load_row(rv, static_cast<const T*>(p.residual), (int32_t)r);
            const T* re = reinterpret_cast<const T*>(rv.w);
#pragma unroll
            for (int j = 0; j < COUT; ++j) acc[j] = fmaf(p.add_scale, elem<T>::to_f32(re[j]), acc[j]);
        }
        if (p.act) {
#pragma unroll
            for (int j = 0; j < COUT; ++j) acc[j] = fmaxf(acc[j], 0.f);
        }
        RowVec<T, COUT> ov;
        T* oe = reinterpret_cast<T*>(ov.w);
#pragma unroll
        for (int j = 0; j < COUT; ++j) oe[j] = elem<T>::from_f32(acc[j]);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + r * COUT);
#pragma unroll
        for (int q = 0; q < RowVec<T, COUT>::kWords; ++q) __stcs(dst + q, ov.w[q]);  // streamed out
    }
}

template <typename T, int CRED, int COUT>
spc_status launch(const GatherGemm& p, cudaStream_t st)
{
    const size_t smem = sizeof(float) * ((size_t)p.K * kSliceStride<CRED, COUT> + COUT);
    auto kern = k_conv_narrow<T, CRED, COUT>;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return SPC_ERR_UNSUPPORTED;
    }
    // resident blocks per SM, looked up once per device and shared-memory size
    static int cached[64][4] = {};
    static size_t cached_smem[64][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPC_ERR_CUDA;
    const int slot = p.K <= 1 ? 0 : (p.K <= 8 ? 1 : (p.K <= 27 ? 2 : 3));
    int per_sm = cached_smem[dev][slot] == smem ? cached[dev][slot] : 0;
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) !=
                cudaSuccess ||
            per_sm < 1)
            return SPC_ERR_UNSUPPORTED;
        cached[dev][slot] = per_sm;
        cached_smem[dev][slot] = smem;
    }
    const int64_t need = ceil_div(p.rows, kThreads);
    const int grid = (int)std::min<int64_t>(need, (int64_t)per_sm * sm_count());
    kern<<<grid, kThreads, smem, st>>>(p);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

template <typename T>
spc_status dispatch(const GatherGemm& p, cudaStream_t st)
{
#define SPC_NARROW_CASE(A, B) \
    if (p.cred == A && p.cout == B) return launch<T, A, B>(p, st);
    SPC_NARROW_CASE(8, 8)
    SPC_NARROW_CASE(8, 16)
    SPC_NARROW_CASE(16, 8)
    SPC_NARROW_CASE(16, 16)
    SPC_NARROW_CASE(16, 32)
    SPC_NARROW_CASE(32, 16)
    SPC_NARROW_CASE(32, 32)
#undef SPC_NARROW_CASE
    return SPC_ERR_UNSUPPORTED;
}

}  // namespace

bool conv_narrow_supported(int32_t cred, int32_t cout, int32_t K, spc_dtype dt)
{
    auto ok = [](int c) { return c == 8 || c == 16 || c == 32; };
    if (!ok(cred) || !ok(cout) || K < 1) return false;
    if (cred == 8 && cout == 32) return false;
    if (cred == 32 && cout == 8) return false;
    // fp32 weights of all offsets must fit in shared memory
    if ((size_t)K * (cred * cout + 4) * sizeof(float) > 200 * 1024) return false;
    (void)dt;
    return true;
}

spc_status conv_gather_narrow(const GatherGemm& p, spc_dtype dt, cudaStream_t st)
{
    if (p.rows == 0) return SPC_OK;
    switch (dt) {
    case SPC_F32: return dispatch<float>(p, st);
    case SPC_F16: return dispatch<__half>(p, st);
    case SPC_BF16: return dispatch<__nv_bfloat16>(p, st);
    }
    return SPC_ERR_INVALID_ARG;
}

}  // namespace spc
