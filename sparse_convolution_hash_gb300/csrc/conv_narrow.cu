// conv_narrow.cu -- gathered conv for narrow channels (Cin, Cout in {8, 16, 32}).
//
// Narrow layers move far more bytes than they compute (a 16 -> 16 pair is 256
// multiply-adds on a 32-byte row), so this path is laid out for memory, not
// for tensor cores: one thread owns one output row and keeps its Cout fp32
// accumulators in registers; the weight tensor is converted to fp32 once per
// persistent block and kept in shared memory.  A warp walks the union of its
// rows' offset masks in a warp-uniform order, so all lanes working on offset k
// read the same W[k] words (shared-memory broadcast), and only lanes whose row
// has a neighbour at k read the map entry and gather the neighbour's row
// (16-byte vector loads).  Rows are written once, with vector stores.
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
#pragma unroll
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

template <typename T, int CRED, int COUT>
__global__ void __launch_bounds__(kThreads) k_conv_narrow(GatherGemm p)
{
    // offsets whose map and row loads are in flight together (about 32 registers of rows)
    constexpr int kRowRegs = CRED * (int)sizeof(T) / 4;
    constexpr int kBatch = kRowRegs >= 32 ? 1 : (kRowRegs >= 16 ? 2 : 4);
    extern __shared__ __align__(16) float s_w[];  // [K][CRED][COUT] fp32, then bias [COUT]
    const T* __restrict__ in = static_cast<const T*>(p.in);
    const int K = p.K;
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
                    int dst = g;
                    if (p.transpose_w) {  // global [K][COUT][CRED] -> shared [K][CRED][COUT]
                        const int k = g / (CRED * COUT), a = (g / CRED) % COUT, b = g % CRED;
                        dst = (k * CRED + b) * COUT + a;
                    }
                    s_w[dst] = elem<T>::to_f32(e[t]);
                }
            }
        }
    }
    float* s_bias = s_w + (size_t)K * CRED * COUT;
    for (int j = threadIdx.x; j < COUT; j += blockDim.x)
        s_bias[j] = p.bias ? elem<T>::to_f32(static_cast<const T*>(p.bias)[j]) : 0.f;
    __syncthreads();

    const uint32_t kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < p.rows; base += step) {
        const int64_t r = base + threadIdx.x;
        const bool valid = r < p.rows;
        float acc[COUT];
#pragma unroll
        for (int j = 0; j < COUT; ++j) acc[j] = s_bias[j];

        if (p.mask) {
            uint32_t m = 0;
            if (valid) {
                m = p.mask[r];
                if (p.mirror) m = __brev(m) >> (32 - K);
                m &= kmask;
            }
            uint32_t todo = __reduce_or_sync(FULL_MASK, m);
            while (todo) {
                // take up to kBatch offsets of the warp's union (warp-uniform)
                int ks[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    ks[b] = todo ? __ffs(todo) - 1 : -1;
                    todo &= todo - 1;
                }
                int32_t idx[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    idx[b] = -1;
                    if (ks[b] >= 0 && ((m >> ks[b]) & 1u)) {
                        const int mk = p.mirror ? K - 1 - ks[b] : ks[b];
                        idx[b] = p.map ? p.map[(int64_t)mk * p.rows + r] : (int32_t)r;
                    }
                }
                RowVec<T, CRED> xv[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (idx[b] >= 0) load_row(xv[b], in, idx[b]);
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (idx[b] >= 0) fma_row<T, CRED, COUT>(acc, xv[b], s_w + (size_t)ks[b] * CRED * COUT);
            }
        } else {
            for (int k = 0; k < K; ++k) {
                int32_t i = -1;
                if (valid) {
                    const int mk = p.mirror ? K - 1 - k : k;
                    i = p.map ? p.map[(int64_t)mk * p.rows + r] : (int32_t)r;
                }
                if (i < 0) continue;
                RowVec<T, CRED> xv;
                load_row(xv, in, i);
                fma_row<T, CRED, COUT>(acc, xv, s_w + (size_t)k * CRED * COUT);
            }
        }
        if (valid) {
            RowVec<T, COUT> ov;
            T* oe = reinterpret_cast<T*>(ov.w);
#pragma unroll
            for (int j = 0; j < COUT; ++j) oe[j] = elem<T>::from_f32(acc[j]);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + r * COUT);
#pragma unroll
            for (int q = 0; q < RowVec<T, COUT>::kWords; ++q) dst[q] = ov.w[q];
        }
    }
}

template <typename T, int CRED, int COUT>
spc_status launch(const GatherGemm& p, cudaStream_t st)
{
    const size_t smem = sizeof(float) * ((size_t)p.K * CRED * COUT + COUT);
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
    if ((size_t)K * cred * cout * sizeof(float) > 200 * 1024) return false;
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
