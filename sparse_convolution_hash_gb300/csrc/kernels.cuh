// kernels.cuh -- internal launch interfaces between the C ABI (api.cu) and the
// kernel translation units.  Everything here is device-side work enqueued on a
// stream; argument validation happens in api.cu before these are called.
#pragma once

#include "common.cuh"

namespace spc {

// Bound (ns) of the waits of one warp role on another in the pipelined
// tensor-core kernels, as set by spc_set_wait_limit_ns (api.cu).
uint64_t wait_limit_ns();

// ------------------------------------------------------------------ hash table
// Open addressing over 32-byte buckets of four 64-bit slots.  A slot holds
// (cell key << vbits) | row, or all ones when empty.  A 4-lane group of a warp
// reads one bucket per step (one L2 sector) and resolves the probe with a
// ballot; buckets are visited linearly from the key's multiplicative hash.
struct HashTable {
    unsigned long long* slots;  // [4 << log2_buckets]
    int log2_buckets;
    int vbits;                  // bits of the row field
};

// Number of 64-bit slots a table for n keys uses (load factor <= 1/2).
int64_t hash_slots_for(int64_t n);

// vbits for n rows, and whether every key of a grid of `cells` cells fits beside it.
int hash_vbits_for(int64_t n);
bool hash_keys_fit(int64_t cells, int vbits);

// Geometry of a probe: the cell read by query row o through offset index
// (a, b, c) is q*stride - pad + (a, b, c)*dil per axis.
struct ProbeGeom {
    int32_t in_shape[3];   // grid of the table's cells
    int32_t q_shape[3];    // grid the query coordinates must lie in
    int32_t ksize[3];
    int32_t stride[3];
    int32_t pad[3];
    int32_t dil[3];
    int32_t batch;
    int32_t K;
    int32_t centre;        // offset index that maps each row to itself (subm), or -1
};

// Buffers a build starts from: each region is filled with a 32-bit pattern.
struct FillRegion {
    uint32_t* p;
    int64_t n;   // 32-bit words
    uint32_t v;
};
struct FillList {
    FillRegion r[5];
};
spc_status build_init(const FillList& L, int n, cudaStream_t st);
// True when the probe fills a submanifold map through offset mirrors (k <= centre).
bool probe_mirror(const ProbeGeom& g, bool with_transpose);
// Per-row fills the insert does for the probe: planes x [stride] int32 set to
// -1 at each inserted row (the mirrored rows of a submanifold map, or the
// transposed map), and mask[row] = 0 when mask is given.
struct RowFill {
    int32_t* p;
    int32_t planes;
    int64_t stride;
    uint32_t* mask;
};
spc_status hash_insert(const int32_t* coords, int64_t n, int32_t batch, const int32_t shape[3],
                       HashTable t, int32_t* status, const RowFill& fill, cudaStream_t st);
spc_status map_probe(const int32_t* qcoords, int64_t nq, int64_t n_in, const ProbeGeom& g,
                     HashTable t, int32_t* imap, int32_t* imap_t, int32_t* pair_count,
                     uint32_t* mask, int32_t* status, cudaStream_t st);

// Sparse max pooling on a strided map (maxpool.cu).
spc_status maxpool_fwd(const void* x, const int32_t* imap, const uint32_t* mask, int32_t K,
                       int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* y, uint8_t* arg,
                       cudaStream_t st);
spc_status maxpool_dgrad(const void* dy, const int32_t* imap_t, const uint8_t* arg, int32_t K,
                         int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* dx,
                         cudaStream_t st);

// Row order of a map grouped by offset mask (rows.cu).
size_t row_order_ws_bytes(int64_t n);
spc_status map_row_order(const int32_t* map, int32_t K, int64_t n, uint32_t* mask, int32_t* perm,
                         void* ws, size_t ws_bytes, cudaStream_t st);
// Stable LSD radix sort of n 64-bit keys on bits [lo_bit, hi_bit) (outcoords.cu);
// keys end in `a` (b is scratch); counter holds n on the device.
size_t radix_ws_bytes(int64_t n);
spc_status radix_sort_keys(unsigned long long* a, unsigned long long* b, const unsigned long long* counter,
                           int64_t n, int lo_bit, int hi_bit, void* ws, cudaStream_t st);

// ------------------------------------------------------ strided output coords
size_t outcoords_ws_bytes(int64_t n_in, int32_t K);
spc_status strided_out_coords(const int32_t* coords, int64_t n_in, const ProbeGeom& g,
                              const int32_t out_shape[3], int32_t* out_coords, int64_t cap,
                              int64_t* n_out, int32_t* status, void* ws, size_t ws_bytes,
                              cudaStream_t st);

// ------------------------------------------------------------------ conv SIMT
// Gathered implicit GEMM on CUDA cores:
//   out[r, j] = bias[j] + sum_k sum_c in[map(k, r), c] * B(k, c, j)
// with map(k, r) = map[mk * rows + r] (mk = k, or K-1-k when mirror), or r when
// map == NULL (K == 1), and B(k, c, j) = w[k][c][j], or w[k][j][c] when
// transpose_w.  `cred` is the reduction width (columns of `in`), `cout` the
// output width; the weight tensor is [K][cred][cout], or [K][cout][cred] when
// transposed.
struct GatherGemm {
    const void* in;
    const void* w;
    const void* bias;
    const int32_t* map;
    const uint32_t* mask;   // per output row, bit k = map(k, r) != -1 (or NULL)
    void* out;
    int64_t rows;           // output rows
    int64_t in_rows;
    int32_t K;
    int32_t cred;
    int32_t cout;
    int32_t mirror;
    int32_t transpose_w;
    // fused epilogue: out = act(acc + bias + add_scale * residual), act 1 = ReLU
    const void* residual;   // [rows, cout] or NULL
    float add_scale;
    int32_t act;
};
spc_status conv_gather_simt(const GatherGemm& p, spc_dtype dt, cudaStream_t st);

// Narrow channels (cred, cout in {8, 16, 32}): one thread per output row.
bool conv_narrow_supported(int32_t cred, int32_t cout, int32_t K, spc_dtype dt);
spc_status conv_gather_narrow(const GatherGemm& p, spc_dtype dt, cudaStream_t st);

// Tensor-core gathered GEMM (tcgen05): out[r, n] = bias[n] + sum_k sum_c
// in[map(k, r), c] * B(k, c, n), with B(k, c, n) = b[k][n][c] (b in
// [K][n_total][cred] order), or b[k][c][n] when b_mn (weights as stored; 16-bit
// types with cred and n_total multiples of 64 only).  wait_ns bounds the waits
// of one warp role on another (SPC_ERR_TIMEOUT when one runs out).
struct TcArgs {
    const void* in;
    const void* b;
    const void* bias;
    const int32_t* map;
    const uint32_t* mask;
    void* out;
    int32_t* status;
    int64_t rows, in_rows;
    int32_t K, cred, n_total, mirror;
    const void* residual;   // fused epilogue, as in GatherGemm
    float add_scale;
    int32_t act;
    const int32_t* perm;    // tile row r computes output row perm[r] (NULL: r)
    int32_t b_mn;
    uint64_t wait_ns;
};
bool conv_tc_supported(int32_t cred, int32_t cout, int32_t K, spc_dtype dt, spc_precision prec);
// True when the forward reads W as stored (no transposed copy in the workspace).
bool conv_tc_reads_w_as_stored(int32_t cin, int32_t cout, spc_dtype dt);
size_t conv_tc_weight_bytes(int32_t K, int32_t cin, int32_t cout, spc_dtype dt);
spc_status transpose_weights(const void* w, void* wt, int32_t K, int32_t cin, int32_t cout,
                             spc_dtype dt, cudaStream_t st);
spc_status conv_gather_tc(const TcArgs& a, spc_dtype dt, cudaStream_t st);

// Quantized forward (conv_i8.cu): int8 codes in and out, exact integer sums on
// the fp16 tensor-core path, per-channel fp32 scale and bias, optional int8
// residual add and ReLU.  wq is the workspace for the split weights.
struct I8Args {
    const int8_t* in;
    __half* wq;
    const float* scale;
    const float* bias;      // or NULL
    const int8_t* add;      // [rows, cout] or NULL
    float add_scale;
    int32_t act;
    const int32_t* map;
    const uint32_t* mask;
    const int32_t* perm;    // tile row r computes output row perm[r] (NULL: r)
    int8_t* out;
    int32_t* status;
    int64_t rows, in_rows;
    int32_t K, cin, cout;
    uint64_t wait_ns;
};
bool conv_i8_supported(int32_t K, int32_t cin, int32_t cout);
size_t conv_i8_ws_bytes(int32_t K, int32_t cin, int32_t cout);
spc_status conv_i8(const I8Args& a, const int8_t* w, cudaStream_t st);

// dW[k] = sum_o x[map[k,o]]^T dy[o] in fp32, deterministic split over output rows.
struct WgradArgs {
    const void* x;
    const void* dy;
    const int32_t* map;
    float* dw;
    int64_t n_in, n_out;
    int32_t K, cin, cout;
};
size_t wgrad_ws_bytes(int32_t K, int64_t n_out, int32_t cin, int32_t cout);
// Fixed-order sum of dfilter partials [K x cin/64 x cout/64 tiles][splits][64][64].
spc_status wgrad_reduce(const float* part, int32_t K, int32_t cin, int32_t cout, int splits,
                        float* dw, cudaStream_t st);

// Tensor-core dfilter: partial 64 x 64 tiles per (offset, channel tile, row split).
struct WgradTcArgs {
    const void* x;
    const void* dy;
    const int32_t* map;
    float* part;            // [tiles][splits][64][64]
    int32_t* status;
    int64_t n_in, n_out;
    int64_t chunk;          // output rows per split (multiple of 128)
    int32_t K, cin, cout, splits;
    uint64_t wait_ns;       // bound of the waits of one warp role on another
};
bool wgrad_tc_supported(int32_t K, int32_t cin, int32_t cout, spc_dtype dt);
int wgrad_tc_splits(int32_t K, int64_t n_out, int32_t cin, int32_t cout);
spc_status wgrad_tc(const WgradTcArgs& a, spc_dtype dt, cudaStream_t st);
spc_status conv_wgrad_simt(const WgradArgs& a, spc_dtype dt, void* ws, size_t ws_bytes,
                           cudaStream_t st);

}  // namespace spc
