// conv_simt.cu -- gathered implicit GEMM on CUDA cores (exact fp32 multiplies).
//
// Output-stationary: a block owns 64 output rows x 64 output channels and walks
// every kernel offset k, gathering the 64 input rows map(k, r) into shared
// memory (absent neighbours read as zero rows) and multiplying them with the
// weight slice W[k].  All offsets accumulate in registers; each output row is
// written once, so there are no atomics and results are run-to-run identical.
// Offsets that no row of the tile uses are skipped.
//
// The same kernel computes dinput: rows are input rows, the map is the
// transposed map (or a submanifold map read through its offset mirror) and the
// weight slice is read transposed.
//
// dfilter: dW[k] = sum over active pairs of x[i]^T dy[o], split over fixed
// chunks of output rows; each (offset, tile, chunk) partial goes to the
// workspace and a second kernel sums the chunks in a fixed order.
#include "kernels.cuh"

namespace spc {

namespace {

constexpr int BM = 64, BN = 64, BK = 32, kThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads) k_gather_gemm_simt(GatherGemm p)
{
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ int32_t s_idx[BM];
    const T* __restrict__ in = static_cast<const T*>(p.in);
    const T* __restrict__ w = static_cast<const T*>(p.w);
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * BM;
    const int col0 = blockIdx.y * BN;
    const int tr = tid >> 4, tc = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

    for (int k = 0; k < p.K; ++k) {
        bool mine = false;
        if (tid < BM) {
            const int64_t r = row0 + tid;
            int32_t i = -1;
            if (r < p.rows) {
                if (p.map) {
                    const int mk = p.mirror ? p.K - 1 - k : k;
                    i = p.map[(int64_t)mk * p.rows + r];
                } else {
                    i = (int32_t)r;
                }
            }
            s_idx[tid] = i;
            mine = i >= 0;
        }
        if (!__syncthreads_or(mine)) continue;
        for (int c0 = 0; c0 < p.cred; c0 += BK) {
            for (int e = tid; e < BM * BK; e += kThreads) {
                const int rr = e / BK, cc = e % BK;
                const int32_t i = s_idx[rr];
                float v = 0.f;
                if (i >= 0 && c0 + cc < p.cred) v = elem<T>::to_f32(in[(int64_t)i * p.cred + c0 + cc]);
                As[cc][rr] = v;
            }
            for (int e = tid; e < BK * BN; e += kThreads) {
                const int cc = e / BN, jj = e % BN;
                const int c = c0 + cc, j = col0 + jj;
                float v = 0.f;
                if (c < p.cred && j < p.cout) {
                    const int64_t off = p.transpose_w ? ((int64_t)k * p.cout + j) * p.cred + c
                                                      : ((int64_t)k * p.cred + c) * p.cout + j;
                    v = elem<T>::to_f32(w[off]);
                }
                Bs[cc][jj] = v;
            }
            __syncthreads();
#pragma unroll 8
            for (int cc = 0; cc < BK; ++cc) {
                float a[4], b[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    a[q] = As[cc][tr * 4 + q];
                    b[q] = Bs[cc][tc * 4 + q];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
            }
            __syncthreads();
        }
    }

    T* __restrict__ out = static_cast<T*>(p.out);
    const T* __restrict__ bias = static_cast<const T*>(p.bias);
    const T* __restrict__ res = static_cast<const T*>(p.residual);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int64_t r = row0 + tr * 4 + x;
        if (r >= p.rows) continue;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int j = col0 + tc * 4 + y;
            if (j >= p.cout) continue;
            float v = acc[x][y];
            if (bias) v += elem<T>::to_f32(bias[j]);
            if (res) v = fmaf(p.add_scale, elem<T>::to_f32(res[r * p.cout + j]), v);
            if (p.act) v = fmaxf(v, 0.f);
            out[r * p.cout + j] = elem<T>::from_f32(v);
        }
    }
}

// ------------------------------------------------------------------- dfilter
constexpr int WT = 64;      // dW tile (cin x cout) per block
constexpr int WO = 32;      // output rows staged per step
constexpr int64_t kChunkRows = 8192;

inline int wgrad_splits(int64_t n_out)
{
    const int64_t s = ceil_div(n_out > 0 ? n_out : 1, kChunkRows);
    return (int)std::min<int64_t>(std::max<int64_t>(s, 1), 64);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
k_wgrad_partial(WgradArgs a, int ctiles, int jtiles, int splits, int64_t chunk,
                float* __restrict__ part)
{
    __shared__ float Xs[WO][WT + 4];
    __shared__ float Gs[WO][WT + 4];
    __shared__ int32_t s_idx[WO];
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const int tile = blockIdx.x;  // (k, ct, jt)
    const int s = blockIdx.y;
    const int jt = tile % jtiles, ct = (tile / jtiles) % ctiles, k = tile / (jtiles * ctiles);
    const int c0 = ct * WT, j0 = jt * WT;
    const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
    const int64_t o_lo = (int64_t)s * chunk;
    const int64_t o_hi = std::min<int64_t>(a.n_out, o_lo + chunk);
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[q][r] = 0.f;

    for (int64_t ob = o_lo; ob < o_hi; ob += WO) {
        bool mine = false;
        if (tid < WO) {
            const int64_t o = ob + tid;
            int32_t i = -1;
            if (o < o_hi) i = a.map ? a.map[(int64_t)k * a.n_out + o] : (int32_t)o;
            s_idx[tid] = i;
            mine = i >= 0;
        }
        if (!__syncthreads_or(mine)) continue;
        for (int e = tid; e < WO * WT; e += kThreads) {
            const int oo = e / WT, cc = e % WT;
            const int32_t i = s_idx[oo];
            float xv = 0.f, gv = 0.f;
            if (i >= 0) {
                if (c0 + cc < a.cin) xv = elem<T>::to_f32(x[(int64_t)i * a.cin + c0 + cc]);
                if (j0 + cc < a.cout) gv = elem<T>::to_f32(dy[(ob + oo) * a.cout + j0 + cc]);
            }
            Xs[oo][cc] = xv;
            Gs[oo][cc] = gv;
        }
        __syncthreads();
#pragma unroll 8
        for (int oo = 0; oo < WO; ++oo) {
            float xa[4], gb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xa[q] = Xs[oo][tr * 4 + q];
                gb[q] = Gs[oo][tc * 4 + q];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[q][r] = fmaf(xa[q], gb[r], acc[q][r]);
        }
        __syncthreads();
    }
    float* dst = part + ((size_t)tile * splits + s) * (WT * WT);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) dst[(tr * 4 + q) * WT + tc * 4 + r] = acc[q][r];
}

// dw[k][c][j] = sum over q = 0, 1, .. splits - 1 (in that order) of the partial
// tiles part[(k, c / WT, j / WT)][q][c % WT][j % WT].  A thread owns four
// consecutive j (one 16-byte load per partial) and keeps eight partial loads in
// flight ahead of its in-order adds, so the result bits do not depend on the
// launch shape.
__global__ void __launch_bounds__(kThreads)
k_wgrad_reduce(const float* __restrict__ part, int K, int cin, int cout, int ctiles, int jtiles,
               int splits, float* __restrict__ dw)
{
    const int64_t total4 = (int64_t)K * cin * cout / 4;  // cout % 4 == 0
    for (int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e4 < total4;
         e4 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = e4 * 4;
        const int j = (int)(e % cout);
        const int c = (int)((e / cout) % cin);
        const int k = (int)(e / ((int64_t)cout * cin));
        const int tile = (k * ctiles + c / WT) * jtiles + j / WT;
        const float4* src = reinterpret_cast<const float4*>(part + (size_t)tile * splits * (WT * WT) +
                                                            (c % WT) * WT + (j % WT));
        constexpr int kStep = WT * WT / 4;  // float4s between successive partials
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        int q = 0;
        for (; q + 8 <= splits; q += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcs(src + (size_t)(q + u) * kStep);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                s.x += v[u].x;
                s.y += v[u].y;
                s.z += v[u].z;
                s.w += v[u].w;
            }
        }
        for (; q < splits; ++q) {
            const float4 v = __ldcs(src + (size_t)q * kStep);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        *reinterpret_cast<float4*>(dw + e) = s;
    }
}

// The same sums one element per thread (any cout).
__global__ void __launch_bounds__(kThreads)
k_wgrad_reduce1(const float* __restrict__ part, int K, int cin, int cout, int ctiles, int jtiles,
                int splits, float* __restrict__ dw)
{
    const int64_t total = (int64_t)K * cin * cout;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % cout);
        const int c = (int)((e / cout) % cin);
        const int k = (int)(e / ((int64_t)cout * cin));
        const int tile = (k * ctiles + c / WT) * jtiles + j / WT;
        const float* src = part + (size_t)tile * splits * (WT * WT) + (c % WT) * WT + (j % WT);
        float s = 0.f;
        for (int q = 0; q < splits; ++q) s += src[(size_t)q * WT * WT];
        dw[e] = s;
    }
}

template <typename T>
spc_status launch_gather(const GatherGemm& p, cudaStream_t st)
{
    dim3 grid((unsigned)ceil_div(p.rows, BM), (unsigned)ceil_div(p.cout, BN));
    k_gather_gemm_simt<T><<<grid, kThreads, 0, st>>>(p);
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

template <typename T>
spc_status launch_wgrad(const WgradArgs& a, void* ws, cudaStream_t st)
{
    const int ctiles = (int)ceil_div(a.cin, WT), jtiles = (int)ceil_div(a.cout, WT);
    const int splits = wgrad_splits(a.n_out);
    const int64_t chunk = ceil_div(ceil_div(a.n_out > 0 ? a.n_out : 1, splits), WO) * WO;
    float* part = static_cast<float*>(ws);
    dim3 grid((unsigned)(a.K * ctiles * jtiles), (unsigned)splits);
    k_wgrad_partial<T><<<grid, kThreads, 0, st>>>(a, ctiles, jtiles, splits, chunk, part);
    SPC_LAUNCH_CHECK();
    return wgrad_reduce(part, a.K, a.cin, a.cout, splits, a.dw, st);
}

}  // namespace

spc_status conv_gather_simt(const GatherGemm& p, spc_dtype dt, cudaStream_t st)
{
    if (p.rows == 0 || p.cout == 0) return SPC_OK;
    switch (dt) {
    case SPC_F32: return launch_gather<float>(p, st);
    case SPC_F16: return launch_gather<__half>(p, st);
    case SPC_BF16: return launch_gather<__nv_bfloat16>(p, st);
    }
    return SPC_ERR_INVALID_ARG;
}

size_t wgrad_ws_bytes(int32_t K, int64_t n_out, int32_t cin, int32_t cout)
{
    const int64_t ctiles = ceil_div(cin, WT), jtiles = ceil_div(cout, WT);
    return sizeof(float) * (size_t)(K * ctiles * jtiles) * (size_t)wgrad_splits(n_out) * WT * WT;
}

spc_status wgrad_reduce(const float* part, int32_t K, int32_t cin, int32_t cout, int splits,
                        float* dw, cudaStream_t st)
{
    const int ctiles = (int)ceil_div(cin, WT), jtiles = (int)ceil_div(cout, WT);
    const int64_t total = (int64_t)K * cin * cout;
    if (total == 0) return SPC_OK;
    if (cout % 4 == 0 && (reinterpret_cast<uintptr_t>(dw) & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(part) & 15u) == 0) {
        const int rgrid = (int)std::min<int64_t>(ceil_div(total / 4, kThreads), 4 * sm_count());
        k_wgrad_reduce<<<rgrid, kThreads, 0, st>>>(part, K, cin, cout, ctiles, jtiles, splits, dw);
    } else {
        const int rgrid = (int)std::min<int64_t>(ceil_div(total, kThreads), 4 * sm_count());
        k_wgrad_reduce1<<<rgrid, kThreads, 0, st>>>(part, K, cin, cout, ctiles, jtiles, splits, dw);
    }
    SPC_LAUNCH_CHECK();
    return SPC_OK;
}

spc_status conv_wgrad_simt(const WgradArgs& a, spc_dtype dt, void* ws, size_t ws_bytes,
                           cudaStream_t st)
{
    if (a.K == 0 || a.cin == 0 || a.cout == 0) return SPC_OK;
    if (!ws || ws_bytes < wgrad_ws_bytes(a.K, a.n_out, a.cin, a.cout)) return SPC_ERR_WORKSPACE;
    switch (dt) {
    case SPC_F32: return launch_wgrad<float>(a, ws, st);
    case SPC_F16: return launch_wgrad<__half>(a, ws, st);
    case SPC_BF16: return launch_wgrad<__nv_bfloat16>(a, ws, st);
    }
    return SPC_ERR_INVALID_ARG;
}

}  // namespace spc
