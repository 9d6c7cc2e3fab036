// api.cu -- the extern "C" entry points of libspc.so declared in include/spc.h.
//
// Each entry point checks its arguments on the host (returning an error before
// anything is enqueued), carves the caller's workspace, and enqueues its
// kernels on the caller's stream.  Nothing here allocates device memory or
// synchronises.
#include <atomic>

#include "kernels.cuh"

using namespace spc;

namespace {
std::atomic<uint64_t> g_wait_ns{2000000000ull};
}  // namespace

uint64_t spc::wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0

bool geom_ok(const spc_geom* g, bool need_stride_pad)
{
    if (!g) return false;
    for (int a = 0; a < 3; ++a) {
        if (g->ksize[a] < 1 || g->dil[a] < 1) return false;
        if (need_stride_pad && (g->stride[a] < 1 || g->pad[a] < 0)) return false;
    }
    return true;
}

int64_t kvol(const spc_geom* g) { return (int64_t)g->ksize[0] * g->ksize[1] * g->ksize[2]; }

bool shape_ok(const int32_t s[3]) { return s && s[0] > 0 && s[1] > 0 && s[2] > 0; }

int32_t axis_out(int32_t in, int32_t k, int32_t s, int32_t p, int32_t dil)
{
    const int64_t span = (int64_t)in + 2 * (int64_t)p - (int64_t)dil * (k - 1) - 1;
    if (span < 0) return 0;
    return (int32_t)(span / s + 1);
}

size_t table_bytes(int64_t n) { return align_up(sizeof(unsigned long long) * (size_t)hash_slots_for(n), 256); }

int elem_bytes(spc_dtype dt) { return dt == SPC_F32 ? 4 : 2; }

bool dtype_ok(spc_dtype dt) { return dt == SPC_F32 || dt == SPC_F16 || dt == SPC_BF16; }

}  // namespace

extern "C" {

const char* spc_status_string(spc_status s)
{
    switch (s) {
    case SPC_OK: return "ok";
    case SPC_ERR_INVALID_ARG: return "invalid argument";
    case SPC_ERR_COORD_RANGE: return "coordinate outside the batch or the grid";
    case SPC_ERR_DUPLICATE: return "duplicate coordinate";
    case SPC_ERR_TABLE_FULL: return "hash table probe bound exceeded";
    case SPC_ERR_CAPACITY: return "output set larger than the output buffer";
    case SPC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SPC_ERR_CUDA: return "CUDA runtime error";
    case SPC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPC_ERR_TIMEOUT: return "an internal GPU wait exceeded its bound";
    }
    return "unknown status";
}

int32_t spc_version(void) { return kVersion; }

spc_status spc_set_wait_limit_ns(uint64_t ns)
{
    if (ns > 60000000000ull) return SPC_ERR_INVALID_ARG;
    g_wait_ns.store(ns, std::memory_order_relaxed);
    return SPC_OK;
}

uint64_t spc_get_wait_limit_ns(void) { return wait_limit_ns(); }

spc_status spc_out_shape(const int32_t in_shape[3], const spc_geom* g, int32_t out_shape[3])
{
    if (!shape_ok(in_shape) || !geom_ok(g, true) || !out_shape) return SPC_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a)
        out_shape[a] = axis_out(in_shape[a], g->ksize[a], g->stride[a], g->pad[a], g->dil[a]);
    return SPC_OK;
}

size_t spc_indice_map_workspace_size(int64_t n_in)
{
    return n_in < 0 ? 0 : table_bytes(n_in);
}

spc_status spc_build_indice_map(const int32_t* coords, int64_t n_in, int32_t batch,
                                const int32_t in_shape[3], const spc_geom* g, int32_t subm,
                                const int32_t* out_coords, int64_t n_out, int32_t* imap,
                                int32_t* imap_t, int32_t* pair_count, uint32_t* mask,
                                int32_t* status, void* ws, size_t ws_bytes, void* stream)
{
    if (n_in < 0 || n_out < 0 || batch < 1 || !shape_ok(in_shape) || !geom_ok(g, !subm))
        return SPC_ERR_INVALID_ARG;
    const int64_t K = kvol(g);
    if (K > (1 << 20)) return SPC_ERR_INVALID_ARG;
    if (!pair_count || !status) return SPC_ERR_INVALID_ARG;
    if (mask && K > 32) return SPC_ERR_INVALID_ARG;
    ProbeGeom pg;
    pg.batch = batch;
    pg.K = (int32_t)K;
    int32_t out_shape[3];
    if (subm) {
        if (n_out != n_in || imap_t) return SPC_ERR_INVALID_ARG;
        for (int a = 0; a < 3; ++a) {
            if (g->ksize[a] % 2 != 1) return SPC_ERR_INVALID_ARG;
            out_shape[a] = in_shape[a];
            pg.stride[a] = 1;
            pg.pad[a] = (g->ksize[a] / 2) * g->dil[a];
        }
        pg.centre = (int32_t)(K / 2);
        out_coords = coords;
    } else {
        for (int a = 0; a < 3; ++a) {
            out_shape[a] = axis_out(in_shape[a], g->ksize[a], g->stride[a], g->pad[a], g->dil[a]);
            pg.stride[a] = g->stride[a];
            pg.pad[a] = g->pad[a];
        }
        pg.centre = -1;
        if (n_out > 0 && !out_coords) return SPC_ERR_INVALID_ARG;
    }
    for (int a = 0; a < 3; ++a) {
        pg.in_shape[a] = in_shape[a];
        pg.q_shape[a] = out_shape[a];
        pg.ksize[a] = g->ksize[a];
        pg.dil[a] = g->dil[a];
    }
    if (n_in > 0 && (!coords || !aligned16(coords))) return SPC_ERR_INVALID_ARG;
    if (n_out > 0 && (!imap || !aligned16(out_coords))) return SPC_ERR_INVALID_ARG;
    if (n_in > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    const unsigned __int128 cells = (unsigned __int128)batch * (unsigned)in_shape[0] *
                                    (unsigned)in_shape[1] * (unsigned)in_shape[2];
    const int vbits = hash_vbits_for(n_in);
    if (cells > (unsigned __int128)INT64_MAX || !hash_keys_fit((int64_t)cells, vbits))
        return SPC_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < spc_indice_map_workspace_size(n_in)) return SPC_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    HashTable t;
    t.slots = static_cast<unsigned long long*>(ws);
    t.log2_buckets = ceil_log2((uint64_t)hash_slots_for(n_in)) - 2;
    t.vbits = vbits;
    // one launch prepares the table and the pair counts; the insert fills, row
    // by row, the buffers indexed by input rows: the transposed map (-1), and
    // for a submanifold map (input rows = output rows) the mirrored map rows
    // (-1) and the mask (0).  A strided map's mask (output rows) goes here too.
    const bool mirror = n_out > 0 && probe_mirror(pg, imap_t != nullptr);
    FillList fl;
    int nf = 0;
    fl.r[nf++] = FillRegion{reinterpret_cast<uint32_t*>(pair_count), K, 0u};
    if (n_out > 0 || n_in > 0) fl.r[nf++] = FillRegion{reinterpret_cast<uint32_t*>(t.slots), (int64_t)8 << t.log2_buckets, 0xFFFFFFFFu};
    if (mask && n_out > 0 && !mirror) fl.r[nf++] = FillRegion{mask, n_out, 0u};
    RowFill rf{nullptr, 0, 0, nullptr};
    if (imap_t && n_in > 0) rf = RowFill{imap_t, (int32_t)K, n_in, nullptr};
    if (mirror) rf = RowFill{imap + (int64_t)(pg.centre + 1) * n_out, (int32_t)(K - pg.centre - 1), n_out, mask};
    spc_status s = build_init(fl, nf, st);
    if (s != SPC_OK) return s;
    if (n_out == 0 && n_in == 0) return SPC_OK;
    if (mirror && n_in == 0) return SPC_OK;
    s = hash_insert(coords, n_in, batch, in_shape, t, status, rf, st);
    if (s != SPC_OK) return s;
    return map_probe(out_coords, n_out, n_in, pg, t, imap, imap_t, pair_count, mask, status, st);
}

size_t spc_strided_out_coords_workspace_size(int64_t n_in, const spc_geom* g)
{
    if (n_in < 0 || !geom_ok(g, true)) return 0;
    return outcoords_ws_bytes(n_in, (int32_t)kvol(g));
}

spc_status spc_strided_out_coords(const int32_t* coords, int64_t n_in, int32_t batch,
                                  const int32_t in_shape[3], const spc_geom* g,
                                  int32_t out_shape[3], int32_t* out_coords, int64_t cap,
                                  int64_t* n_out, int32_t* status, void* ws, size_t ws_bytes,
                                  void* stream)
{
    if (n_in < 0 || cap < 0 || batch < 1 || !shape_ok(in_shape) || !geom_ok(g, true) ||
        !out_shape || !n_out || !status)
        return SPC_ERR_INVALID_ARG;
    const int64_t K = kvol(g);
    if (K > (1 << 20)) return SPC_ERR_INVALID_ARG;
    if (n_in > 0 && (!coords || !aligned16(coords))) return SPC_ERR_INVALID_ARG;
    if (cap > 0 && (!out_coords || !aligned16(out_coords))) return SPC_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a)
        out_shape[a] = axis_out(in_shape[a], g->ksize[a], g->stride[a], g->pad[a], g->dil[a]);
    if (n_in * K > (int64_t)UINT32_MAX) return SPC_ERR_UNSUPPORTED;
    const unsigned __int128 out_cells = (unsigned __int128)batch * (unsigned)out_shape[0] *
                                        (unsigned)out_shape[1] * (unsigned)out_shape[2];
    if (out_cells > (unsigned __int128)INT64_MAX) return SPC_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < spc_strided_out_coords_workspace_size(n_in, g)) return SPC_ERR_WORKSPACE;
    ProbeGeom pg;
    for (int a = 0; a < 3; ++a) {
        pg.in_shape[a] = in_shape[a];
        pg.q_shape[a] = out_shape[a];
        pg.ksize[a] = g->ksize[a];
        pg.stride[a] = g->stride[a];
        pg.pad[a] = g->pad[a];
        pg.dil[a] = g->dil[a];
    }
    pg.batch = batch;
    pg.K = (int32_t)K;
    pg.centre = -1;
    return strided_out_coords(coords, n_in, pg, out_shape, out_coords, cap, n_out, status, ws,
                              ws_bytes, static_cast<cudaStream_t>(stream));
}

size_t spc_conv_workspace_size(int32_t K, int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                               spc_dtype dt)
{
    (void)n_in;
    (void)n_out;
    if (K < 1 || cin < 1 || cout < 1 || !dtype_ok(dt)) return 0;
    // the tensor-core forward needs a transposed copy of the weights unless it
    // reads them as stored
    if ((conv_tc_supported(cin, cout, K, dt, SPC_PREC_EXACT) ||
         conv_tc_supported(cin, cout, K, dt, SPC_PREC_TF32)) &&
        !conv_tc_reads_w_as_stored(cin, cout, dt))
        return conv_tc_weight_bytes(K, cin, cout, dt);
    return 0;
}

namespace {

spc_status check_conv(const void* a, const void* w, const void* out, int32_t K, int64_t n_a,
                      int64_t n_out, int32_t cin, int32_t cout, spc_dtype dt)
{
    if (!dtype_ok(dt) || K < 1 || n_a < 0 || n_out < 0 || cin < 1 || cout < 1)
        return SPC_ERR_INVALID_ARG;
    if (!w || !aligned16(w)) return SPC_ERR_INVALID_ARG;
    if (n_a > 0 && (!a || !aligned16(a))) return SPC_ERR_INVALID_ARG;
    if (n_out > 0 && (!out || !aligned16(out))) return SPC_ERR_INVALID_ARG;
    if (n_a > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    (void)elem_bytes;
    return SPC_OK;
}

// Picks the conv kernel for a gathered GEMM on CUDA cores: the narrow-channel
// kernel when the channel widths allow it, else the general tiled kernel.
spc_status run_gather(const GatherGemm& p, spc_dtype dt, cudaStream_t st)
{
    if (conv_narrow_supported(p.cred, p.cout, p.K, dt) && aligned16(p.in) && aligned16(p.out)) {
        const spc_status s = conv_gather_narrow(p, dt, st);
        if (s != SPC_ERR_UNSUPPORTED) return s;
    }
    return conv_gather_simt(p, dt, st);
}

}  // namespace

namespace {
// The forward of every entry point; perm (or NULL) orders the tensor-core
// kernel's tiles (the CUDA-core kernels own one row per thread and ignore it).
spc_status conv_fwd_impl(const void* x, const void* w, const void* bias, const int32_t* imap,
                         const uint32_t* mask, const int32_t* perm, int32_t K, int64_t n_in,
                         int64_t n_out, int32_t cin, int32_t cout, spc_dtype dt, spc_precision prec,
                         const void* residual, float add_scale, spc_activation act, void* y,
                         int32_t* status, void* ws, size_t ws_bytes, void* stream)
{
    spc_status s = check_conv(x, w, y, K, n_in, n_out, cin, cout, dt);
    if (s != SPC_OK) return s;
    if (act != SPC_ACT_NONE && act != SPC_ACT_RELU) return SPC_ERR_INVALID_ARG;
    if (residual && (!aligned16(residual) || residual == y)) return SPC_ERR_INVALID_ARG;
    if (prec != SPC_PREC_EXACT && prec != SPC_PREC_TF32) return SPC_ERR_INVALID_ARG;
    if (!imap && n_out > 0 && !(K == 1 && n_in == n_out)) return SPC_ERR_INVALID_ARG;
    if (mask && K > 32) return SPC_ERR_INVALID_ARG;
    GatherGemm p;
    p.in = x;
    p.w = w;
    p.bias = bias;
    p.map = imap;
    p.mask = mask;
    p.out = y;
    p.rows = n_out;
    p.in_rows = n_in;
    p.K = K;
    p.cred = cin;
    p.cout = cout;
    p.mirror = 0;
    p.transpose_w = 0;
    p.residual = residual;
    p.add_scale = add_scale;
    p.act = (int32_t)act;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // channel widths of 8 / 16 / 32 on both sides: the latency-oriented CUDA-core
    // kernel (a row has few neighbours on sparse scenes; a tensor-core tile
    // would mostly multiply zero-filled rows)
    const bool narrow = conv_narrow_supported(cin, cout, K, dt);
    if (n_out > 0 && !narrow && conv_tc_supported(cin, cout, K, dt, prec) && aligned16(x) && aligned16(y)) {
        // 16-bit rows of multiples of 64 channels read W[k] as stored (an
        // MN-major operand); the other shapes take it transposed in the workspace
        const bool b_mn = conv_tc_reads_w_as_stored(cin, cout, dt);
        if (!b_mn) {
            const size_t wbytes = conv_tc_weight_bytes(K, cin, cout, dt);
            if (!ws || ws_bytes < wbytes || (reinterpret_cast<uintptr_t>(ws) & 255u))
                return SPC_ERR_WORKSPACE;
            s = transpose_weights(w, ws, K, cin, cout, dt, st);
            if (s != SPC_OK) return s;
        }
        TcArgs a;
        a.in = x;
        a.b = b_mn ? w : ws;
        a.bias = bias;
        a.map = imap;
        a.mask = mask;
        a.out = y;
        a.status = status;
        a.rows = n_out;
        a.in_rows = n_in;
        a.K = K;
        a.cred = cin;
        a.n_total = cout;
        a.mirror = 0;
        a.perm = perm;
        a.residual = residual;
        a.add_scale = add_scale;
        a.act = (int32_t)act;
        a.b_mn = b_mn ? 1 : 0;
        a.wait_ns = wait_limit_ns();
        s = conv_gather_tc(a, dt, st);
        if (s != SPC_ERR_UNSUPPORTED) return s;
    }
    return run_gather(p, dt, st);
}

}  // namespace

spc_status spc_conv_fwd_fused(const void* x, const void* w, const void* bias, const int32_t* imap,
                              const uint32_t* mask, const int32_t* perm, int32_t K, int64_t n_in,
                              int64_t n_out, int32_t cin, int32_t cout, spc_dtype dt,
                              spc_precision prec, const void* residual, float add_scale,
                              spc_activation act, void* y, int32_t* status, void* ws,
                              size_t ws_bytes, void* stream)
{
    if (perm && K > 32) return SPC_ERR_INVALID_ARG;
    return conv_fwd_impl(x, w, bias, imap, mask, perm, K, n_in, n_out, cin, cout, dt, prec,
                         residual, add_scale, act, y, status, ws, ws_bytes, stream);
}

spc_status spc_conv_fwd(const void* x, const void* w, const void* bias, const int32_t* imap,
                        const uint32_t* mask, int32_t K, int64_t n_in, int64_t n_out, int32_t cin,
                        int32_t cout, spc_dtype dt, spc_precision prec, void* y, int32_t* status,
                        void* ws, size_t ws_bytes, void* stream)
{
    return conv_fwd_impl(x, w, bias, imap, mask, nullptr, K, n_in, n_out, cin, cout, dt, prec,
                         nullptr, 0.f, SPC_ACT_NONE, y, status, ws, ws_bytes, stream);
}

size_t spc_conv_int8_workspace_size(int32_t K, int32_t cin, int32_t cout)
{
    if (!conv_i8_supported(K, cin, cout)) return 0;
    return conv_i8_ws_bytes(K, cin, cout);
}

spc_status spc_conv_fwd_int8(const int8_t* x, const int8_t* w, const float* scale,
                             const float* bias, const int32_t* imap, const uint32_t* mask,
                             const int32_t* perm, int32_t K, int64_t n_in, int64_t n_out,
                             int32_t cin, int32_t cout, const int8_t* add, float add_scale,
                             spc_activation act, int8_t* y, int32_t* status, void* ws,
                             size_t ws_bytes, void* stream)
{
    if (K < 1 || n_in < 0 || n_out < 0 || cin < 1 || cout < 1) return SPC_ERR_INVALID_ARG;
    if (act != SPC_ACT_NONE && act != SPC_ACT_RELU) return SPC_ERR_INVALID_ARG;
    if (!w || !aligned16(w) || !scale) return SPC_ERR_INVALID_ARG;
    if (n_in > 0 && (!x || !aligned16(x))) return SPC_ERR_INVALID_ARG;
    if (n_out > 0 && (!y || !aligned16(y))) return SPC_ERR_INVALID_ARG;
    if (add && (!aligned16(add) || add == y)) return SPC_ERR_INVALID_ARG;
    if (!imap && n_out > 0 && !(K == 1 && n_in == n_out)) return SPC_ERR_INVALID_ARG;
    if ((mask || perm) && K > 32) return SPC_ERR_INVALID_ARG;
    if (n_in > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    if (!conv_i8_supported(K, cin, cout)) return SPC_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < conv_i8_ws_bytes(K, cin, cout) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return SPC_ERR_WORKSPACE;
    I8Args a;
    a.in = x;
    a.wq = static_cast<__half*>(ws);
    a.scale = scale;
    a.bias = bias;
    a.add = add;
    a.add_scale = add_scale;
    a.act = (int32_t)act;
    a.map = imap;
    a.mask = mask;
    a.perm = perm;
    a.out = y;
    a.status = status;
    a.rows = n_out;
    a.in_rows = n_in;
    a.K = K;
    a.cin = cin;
    a.cout = cout;
    a.wait_ns = wait_limit_ns();
    return conv_i8(a, w, static_cast<cudaStream_t>(stream));
}

size_t spc_map_row_order_workspace_size(int64_t n) { return n < 0 ? 0 : row_order_ws_bytes(n); }

spc_status spc_map_row_order(const int32_t* map, int32_t K, int64_t n, uint32_t* mask,
                             int32_t* perm, void* ws, size_t ws_bytes, void* stream)
{
    if (K < 1 || K > 32 || n < 0) return SPC_ERR_INVALID_ARG;
    if (n > 0 && ((!map && !mask) || !perm)) return SPC_ERR_INVALID_ARG;
    if (n > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    return map_row_order(map, K, n, mask, perm, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

spc_status spc_maxpool_fwd(const void* x, const int32_t* imap, const uint32_t* mask, int32_t K,
                           int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* y,
                           uint8_t* arg, void* stream)
{
    if (K < 1 || K > 254 || n_in < 0 || n_out < 0 || c < 0 || !dtype_ok(dt)) return SPC_ERR_INVALID_ARG;
    if (mask && K > 32) return SPC_ERR_INVALID_ARG;
    if (n_out > 0 && c > 0 && (!imap || !y || (n_in > 0 && !x))) return SPC_ERR_INVALID_ARG;
    if (n_in > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    return maxpool_fwd(x, imap, mask, K, n_in, n_out, c, dt, y, arg, static_cast<cudaStream_t>(stream));
}

spc_status spc_maxpool_dgrad(const void* dy, const int32_t* imap_t, const uint8_t* arg, int32_t K,
                             int64_t n_in, int64_t n_out, int32_t c, spc_dtype dt, void* dx,
                             void* stream)
{
    if (K < 1 || K > 254 || n_in < 0 || n_out < 0 || c < 0 || !dtype_ok(dt)) return SPC_ERR_INVALID_ARG;
    if (n_in > 0 && c > 0 && (!imap_t || !dx || (n_out > 0 && (!dy || !arg)))) return SPC_ERR_INVALID_ARG;
    if (n_in > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    return maxpool_dgrad(dy, imap_t, arg, K, n_in, n_out, c, dt, dx, static_cast<cudaStream_t>(stream));
}

spc_status spc_conv_inverse(const void* y, const void* w, const void* bias, const int32_t* imap_t,
                            const uint32_t* mask_t, const int32_t* perm, int32_t K, int64_t n_y,
                            int64_t n_out, int32_t cy, int32_t cout, spc_dtype dt,
                            spc_precision prec, void* out, int32_t* status, void* ws,
                            size_t ws_bytes, void* stream)
{
    // the inverse conv gathers through the transposed map: rows of the strided
    // conv's input set are its outputs, rows of its output set its inputs
    if (n_out > 0 && !imap_t) return SPC_ERR_INVALID_ARG;
    if ((mask_t || perm) && K > 32) return SPC_ERR_INVALID_ARG;
    return conv_fwd_impl(y, w, bias, imap_t, mask_t, perm, K, n_y, n_out, cy, cout, dt, prec,
                         nullptr, 0.f, SPC_ACT_NONE, out, status, ws, ws_bytes, stream);
}

spc_status spc_conv_dgrad(const void* dy, const void* w, const int32_t* map, spc_map_kind kind,
                          const uint32_t* mask, const int32_t* perm, int32_t K, int64_t n_in,
                          int64_t n_out, int32_t cin, int32_t cout, spc_dtype dt,
                          spc_precision prec, void* dx, int32_t* status, void* ws,
                          size_t ws_bytes, void* stream)
{
    (void)ws;
    (void)ws_bytes;
    spc_status s = check_conv(dy, w, dx, K, n_out, n_in, cin, cout, dt);
    if (s != SPC_OK) return s;
    if (prec != SPC_PREC_EXACT && prec != SPC_PREC_TF32) return SPC_ERR_INVALID_ARG;
    if (kind != SPC_MAP_TRANSPOSED && kind != SPC_MAP_SUBM_MIRROR) return SPC_ERR_INVALID_ARG;
    if (kind == SPC_MAP_SUBM_MIRROR && n_in != n_out) return SPC_ERR_INVALID_ARG;
    if (!map && n_in > 0 && !(K == 1 && n_in == n_out)) return SPC_ERR_INVALID_ARG;
    if ((mask || perm) && K > 32) return SPC_ERR_INVALID_ARG;
    GatherGemm p;
    p.in = dy;
    p.w = w;
    p.bias = nullptr;
    p.map = map;
    p.mask = mask;
    p.out = dx;
    p.rows = n_in;
    p.in_rows = n_out;
    p.K = K;
    p.cred = cout;
    p.cout = cin;
    p.mirror = (kind == SPC_MAP_SUBM_MIRROR) ? 1 : 0;
    p.transpose_w = 1;
    p.residual = nullptr;
    p.add_scale = 0.f;
    p.act = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool narrow = conv_narrow_supported(cout, cin, K, dt);
    if (n_in > 0 && !narrow && conv_tc_supported(cout, cin, K, dt, prec) && aligned16(dy) && aligned16(dx)) {
        // W[k] is [Cin][Cout]: already the [N][K] K-major operand of dx = dy W[k]^T
        TcArgs a;
        a.in = dy;
        a.b = w;
        a.bias = nullptr;
        a.map = map;
        a.mask = mask;
        a.out = dx;
        a.status = status;
        a.rows = n_in;
        a.in_rows = n_out;
        a.K = K;
        a.cred = cout;
        a.n_total = cin;
        a.mirror = p.mirror;
        a.perm = perm;
        a.residual = nullptr;
        a.add_scale = 0.f;
        a.act = 0;
        a.b_mn = 0;
        a.wait_ns = wait_limit_ns();
        const spc_status s2 = conv_gather_tc(a, dt, st);
        if (s2 != SPC_ERR_UNSUPPORTED) return s2;
    }
    return run_gather(p, dt, st);
}

namespace {
size_t wgrad_tc_ws_bytes(int32_t K, int64_t n_out, int32_t cin, int32_t cout)
{
    const int splits = wgrad_tc_splits(K, n_out, cin, cout);
    return sizeof(float) * (size_t)K * (size_t)(cin / 64) * (size_t)(cout / 64) * (size_t)splits * 4096;
}
}  // namespace

size_t spc_conv_wgrad_workspace_size(int32_t K, int64_t n_in, int64_t n_out, int32_t cin,
                                     int32_t cout, spc_dtype dt)
{
    (void)n_in;
    if (K < 1 || n_out < 0 || cin < 1 || cout < 1) return 0;
    size_t b = wgrad_ws_bytes(K, n_out, cin, cout);
    if (wgrad_tc_supported(K, cin, cout, dt)) b = std::max(b, wgrad_tc_ws_bytes(K, n_out, cin, cout));
    return b;
}

spc_status spc_conv_wgrad(const void* x, const void* dy, const int32_t* imap, int32_t K,
                          int64_t n_in, int64_t n_out, int32_t cin, int32_t cout, spc_dtype dt,
                          spc_precision prec, float* dw, int32_t* status, void* ws,
                          size_t ws_bytes, void* stream)
{
    if (!dtype_ok(dt) || K < 1 || n_in < 0 || n_out < 0 || cin < 1 || cout < 1 || !dw)
        return SPC_ERR_INVALID_ARG;
    if (n_in > 0 && (!x || !aligned16(x))) return SPC_ERR_INVALID_ARG;
    if (n_out > 0 && (!dy || !aligned16(dy))) return SPC_ERR_INVALID_ARG;
    if (n_in > INT32_MAX - 1 || n_out > INT32_MAX - 1) return SPC_ERR_UNSUPPORTED;
    if (prec != SPC_PREC_EXACT && prec != SPC_PREC_TF32) return SPC_ERR_INVALID_ARG;
    if (!imap && n_out > 0 && !(K == 1 && n_in == n_out)) return SPC_ERR_INVALID_ARG;
    if (ws_bytes < spc_conv_wgrad_workspace_size(K, n_in, n_out, cin, cout, dt) || !ws)
        return SPC_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (imap && n_out > 0 && n_in > 0 && wgrad_tc_supported(K, cin, cout, dt) &&
        (reinterpret_cast<uintptr_t>(ws) & 15u) == 0) {
        WgradTcArgs t;
        t.x = x;
        t.dy = dy;
        t.map = imap;
        t.part = static_cast<float*>(ws);
        t.status = status;
        t.n_in = n_in;
        t.n_out = n_out;
        t.K = K;
        t.cin = cin;
        t.cout = cout;
        t.splits = wgrad_tc_splits(K, n_out, cin, cout);
        t.chunk = ceil_div(ceil_div(n_out, t.splits), 128) * 128;
        t.splits = (int)ceil_div(n_out, t.chunk);
        t.wait_ns = wait_limit_ns();
        spc_status s2 = wgrad_tc(t, dt, st);
        if (s2 == SPC_OK) return wgrad_reduce(t.part, K, cin, cout, t.splits, dw, st);
        if (s2 != SPC_ERR_UNSUPPORTED) return s2;
    }
    WgradArgs a;
    a.x = x;
    a.dy = dy;
    a.map = imap;
    a.dw = dw;
    a.n_in = n_in;
    a.n_out = n_out;
    a.K = K;
    a.cin = cin;
    a.cout = cout;
    return conv_wgrad_simt(a, dt, ws, ws_bytes, st);
}

}  // extern "C"
