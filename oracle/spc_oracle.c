/*
 * spc_oracle.c -- plain, slow CPU oracle for sparse 3-D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may call this file:
 * only the test suite, the package smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (all from the method's definitions, in the plainest order):
 *
 *  - Coordinates are rows (b, z, y, x) of int32, batch first, as in spconv's
 *    SparseConvTensor ("spconv.pytorch Core Concepts Definitions", USAGE.md).
 *  - Kernel offsets are taken in C order over (kz, ky, kx); for a submanifold
 *    conv the offset of index (a, b, c) is ((a - kz/2) dil_z, (b - ky/2) dil_y,
 *    (c - kx/2) dil_x), centred, as in lato_mlx sparse/conv.py
 *    "_kernel_offsets" (C order over (dz, dy, dx), spconv's ordering).
 *  - Submanifold map: output set = input set; imap[k, o] is the input row at
 *    coords[o] + d_k when that cell is occupied and in the grid, else -1
 *    (lato_mlx conv.py, "build_indice_map" docstring and the module docstring's
 *    formula out[c] = bias + sum_d W[d] @ feats[c + d] over occupied c + d).
 *    Found by binary search over the sorted key set, one lookup per (o, k).
 *  - Strided (regular) sparse conv: its result is that of a dense conv run on
 *    the densified tensor, evaluated only where input data exists (spconv
 *    USAGE.md, "Core Concepts Definitions", Sparse Convolution).  Output grid
 *    size per axis is the dense conv's,
 *    floor((in + 2p - dil (k-1) - 1) / s) + 1; output o reads input
 *    i = o s - p + k dil; the output set is every output cell whose receptive
 *    field holds at least one occupied input (cells outside the output grid are
 *    dropped, spconv COMMON_PROBLEMS.md, the [8,200,200] k3 s2 p[0,1,1]
 *    example whose only point z=7 yields no output).  Output rows are sorted
 *    by (b, z, y, x).
 *  - Forward:  y[o, :] = bias + sum_k sum_{i = imap[k,o] != -1} x[i, :] W[k],
 *    W laid out [K, Cin, Cout] (lato_mlx conv.py, SubMConv3d).
 *  - dinput:   dx[i, :] = sum over pairs (k, o) with imap[k,o] = i of W[k] dy[o, :].
 *  - dfilter:  dW[k] = sum over o with imap[k,o] = i != -1 of x[i, :]^T dy[o, :].
 *    (both are the gradients of the forward sum; "dinput"/"dfilter" as named in
 *    the HYGON-AI spconv-das README, Testing and Accuracy.)
 *
 * All floating point is double precision on the exact input values.
 *
 * Output rows are independent, so the row loops of the map probe, the forward
 * and the max pool run as OpenMP parallel loops when the file is compiled with
 * OpenMP (each row is still computed by one thread in the order written, so the
 * results do not depend on the thread count); orc_set_threads picks the count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_RANGE 1
#define ORC_ERR_DUPLICATE 2
#define ORC_ERR_ARG 3
#define ORC_ERR_CAPACITY 4
#define ORC_ERR_NOMEM 5

typedef struct {
    int64_t key;
    int64_t row;
} orc_entry;

/* Threads of the parallel row loops (n > 0 sets them); returns the count in
 * effect, 1 without OpenMP. */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

static int cmp_entry(const void* a, const void* b)
{
    int64_t ka = ((const orc_entry*)a)->key, kb = ((const orc_entry*)b)->key;
    return (ka > kb) - (ka < kb);
}

static int cmp_i64(const void* a, const void* b)
{
    int64_t ka = *(const int64_t*)a, kb = *(const int64_t*)b;
    return (ka > kb) - (ka < kb);
}

/* Mixed-radix key of a cell over a (batch, D, H, W) grid. */
static int64_t cell_key(int64_t b, int64_t z, int64_t y, int64_t x, const int32_t shape[3])
{
    return ((b * shape[0] + z) * shape[1] + y) * shape[2] + x;
}

static int in_grid(int64_t z, int64_t y, int64_t x, const int32_t shape[3])
{
    return z >= 0 && z < shape[0] && y >= 0 && y < shape[1] && x >= 0 && x < shape[2];
}

/* Sorted (key, row) table of a coordinate set; rejects out-of-range and duplicate rows. */
static int sorted_set(const int32_t* coords, int64_t n, int32_t batch, const int32_t shape[3],
                      orc_entry** out)
{
    orc_entry* e = (orc_entry*)malloc(sizeof(orc_entry) * (size_t)(n > 0 ? n : 1));
    if (!e) return ORC_ERR_NOMEM;
    for (int64_t r = 0; r < n; ++r) {
        const int32_t* c = coords + 4 * r;
        if (c[0] < 0 || c[0] >= batch || !in_grid(c[1], c[2], c[3], shape)) {
            free(e);
            return ORC_ERR_RANGE;
        }
        e[r].key = cell_key(c[0], c[1], c[2], c[3], shape);
        e[r].row = r;
    }
    qsort(e, (size_t)n, sizeof(orc_entry), cmp_entry);
    for (int64_t r = 1; r < n; ++r) {
        if (e[r].key == e[r - 1].key) {
            free(e);
            return ORC_ERR_DUPLICATE;
        }
    }
    *out = e;
    return ORC_OK;
}

/* Row of `key` in the sorted table, or -1. */
static int64_t lookup(const orc_entry* e, int64_t n, int64_t key)
{
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (e[mid].key < key) lo = mid + 1;
        else hi = mid;
    }
    return (lo < n && e[lo].key == key) ? e[lo].row : -1;
}

/* Kernel index k -> (a, b, c) in C order over (kz, ky, kx). */
static void kernel_index(int64_t k, const int32_t ksize[3], int64_t abc[3])
{
    abc[2] = k % ksize[2];
    abc[1] = (k / ksize[2]) % ksize[1];
    abc[0] = k / ((int64_t)ksize[2] * ksize[1]);
}

static int check_geom(const int32_t ksize[3], const int32_t dil[3])
{
    for (int a = 0; a < 3; ++a)
        if (ksize[a] < 1 || dil[a] < 1) return ORC_ERR_ARG;
    return ORC_OK;
}

int orc_subm_map(const int32_t* coords, int64_t n, int32_t batch, const int32_t shape[3],
                 const int32_t ksize[3], const int32_t dil[3], int32_t* imap, int64_t* pair_count)
{
    if (check_geom(ksize, dil) != ORC_OK || n < 0 || batch < 1) return ORC_ERR_ARG;
    for (int a = 0; a < 3; ++a)
        if (ksize[a] % 2 != 1) return ORC_ERR_ARG;
    const int64_t K = (int64_t)ksize[0] * ksize[1] * ksize[2];
    orc_entry* e = NULL;
    int st = sorted_set(coords, n, batch, shape, &e);
    if (st != ORC_OK) return st;
    for (int64_t k = 0; k < K; ++k) {
        int64_t abc[3];
        kernel_index(k, ksize, abc);
        int64_t d[3];
        for (int a = 0; a < 3; ++a) d[a] = (abc[a] - ksize[a] / 2) * dil[a];
        int64_t hits = 0;
#pragma omp parallel for schedule(static) reduction(+ : hits)
        for (int64_t o = 0; o < n; ++o) {
            const int32_t* c = coords + 4 * o;
            int64_t z = c[1] + d[0], y = c[2] + d[1], x = c[3] + d[2];
            int64_t row = -1;
            if (in_grid(z, y, x, shape)) row = lookup(e, n, cell_key(c[0], z, y, x, shape));
            imap[k * n + o] = (int32_t)row;
            hits += row >= 0;
        }
        pair_count[k] = hits;
    }
    free(e);
    return ORC_OK;
}

/* Dense-conv output extent along one axis (0 when the window never fits). */
static int32_t axis_out(int32_t in, int32_t k, int32_t s, int32_t p, int32_t dil)
{
    int64_t span = (int64_t)in + 2 * (int64_t)p - (int64_t)dil * (k - 1) - 1;
    if (span < 0) return 0;
    return (int32_t)(span / s + 1);
}

int orc_out_shape(const int32_t in_shape[3], const int32_t ksize[3], const int32_t stride[3],
                  const int32_t pad[3], const int32_t dil[3], int32_t out_shape[3])
{
    if (check_geom(ksize, dil) != ORC_OK) return ORC_ERR_ARG;
    for (int a = 0; a < 3; ++a) {
        if (stride[a] < 1 || pad[a] < 0 || in_shape[a] < 1) return ORC_ERR_ARG;
        out_shape[a] = axis_out(in_shape[a], ksize[a], stride[a], pad[a], dil[a]);
    }
    return ORC_OK;
}

int orc_strided_out_coords(const int32_t* coords, int64_t n, int32_t batch, const int32_t in_shape[3],
                           const int32_t ksize[3], const int32_t stride[3], const int32_t pad[3],
                           const int32_t dil[3], int32_t* out_coords, int64_t cap, int64_t* n_out)
{
    int32_t out_shape[3];
    int st = orc_out_shape(in_shape, ksize, stride, pad, dil, out_shape);
    if (st != ORC_OK) return st;
    *n_out = 0;
    orc_entry* e = NULL;
    st = sorted_set(coords, n, batch, in_shape, &e);
    if (st != ORC_OK) return st;
    free(e);
    const int64_t K = (int64_t)ksize[0] * ksize[1] * ksize[2];
    /* every (input, offset) pair that lands on an output cell names that cell */
    int64_t ncand = 0;
    int64_t* cand = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n * K > 0 ? n * K : 1));
    if (!cand) return ORC_ERR_NOMEM;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + 4 * i;
        for (int64_t k = 0; k < K; ++k) {
            int64_t abc[3], o[3];
            kernel_index(k, ksize, abc);
            int ok = 1;
            for (int a = 0; a < 3 && ok; ++a) {
                /* i = o s - p + k dil  <=>  o = (i + p - k dil) / s, when exact */
                int64_t t = (int64_t)c[1 + a] + pad[a] - abc[a] * dil[a];
                if (t < 0 || t % stride[a] != 0) ok = 0;
                else {
                    o[a] = t / stride[a];
                    if (o[a] >= out_shape[a]) ok = 0;
                }
            }
            if (ok) cand[ncand++] = cell_key(c[0], o[0], o[1], o[2], out_shape);
        }
    }
    qsort(cand, (size_t)ncand, sizeof(int64_t), cmp_i64);
    int64_t u = 0;
    for (int64_t j = 0; j < ncand; ++j)
        if (j == 0 || cand[j] != cand[j - 1]) cand[u++] = cand[j];
    *n_out = u;
    if (u > cap) {
        free(cand);
        return ORC_ERR_CAPACITY;
    }
    for (int64_t j = 0; j < u; ++j) {
        int64_t key = cand[j];
        out_coords[4 * j + 3] = (int32_t)(key % out_shape[2]);
        key /= out_shape[2];
        out_coords[4 * j + 2] = (int32_t)(key % out_shape[1]);
        key /= out_shape[1];
        out_coords[4 * j + 1] = (int32_t)(key % out_shape[0]);
        out_coords[4 * j + 0] = (int32_t)(key / out_shape[0]);
    }
    free(cand);
    return ORC_OK;
}

int orc_strided_map(const int32_t* coords, int64_t n, const int32_t* out_coords, int64_t n_out,
                    int32_t batch, const int32_t in_shape[3], const int32_t ksize[3],
                    const int32_t stride[3], const int32_t pad[3], const int32_t dil[3],
                    int32_t* imap, int32_t* imap_t, int64_t* pair_count)
{
    int32_t out_shape[3];
    int st = orc_out_shape(in_shape, ksize, stride, pad, dil, out_shape);
    if (st != ORC_OK) return st;
    const int64_t K = (int64_t)ksize[0] * ksize[1] * ksize[2];
    orc_entry* e = NULL;
    st = sorted_set(coords, n, batch, in_shape, &e);
    if (st != ORC_OK) return st;
    for (int64_t o = 0; o < n_out; ++o) {
        const int32_t* c = out_coords + 4 * o;
        if (c[0] < 0 || c[0] >= batch || !in_grid(c[1], c[2], c[3], out_shape)) {
            free(e);
            return ORC_ERR_RANGE;
        }
    }
    if (imap_t)
        for (int64_t j = 0; j < K * n; ++j) imap_t[j] = -1;
    for (int64_t k = 0; k < K; ++k) {
        int64_t abc[3];
        kernel_index(k, ksize, abc);
        int64_t hits = 0;
        for (int64_t o = 0; o < n_out; ++o) {
            const int32_t* c = out_coords + 4 * o;
            int64_t p[3];
            for (int a = 0; a < 3; ++a) p[a] = (int64_t)c[1 + a] * stride[a] - pad[a] + abc[a] * dil[a];
            int64_t row = -1;
            if (in_grid(p[0], p[1], p[2], in_shape))
                row = lookup(e, n, cell_key(c[0], p[0], p[1], p[2], in_shape));
            imap[k * n_out + o] = (int32_t)row;
            if (row >= 0) {
                ++hits;
                if (imap_t) imap_t[k * n + row] = (int32_t)o;
            }
        }
        pair_count[k] = hits;
    }
    free(e);
    return ORC_OK;
}

/* imap_t[k, i] = o for every pair imap[k, o] = i; -1 elsewhere. */
void orc_transpose_map(const int32_t* imap, int64_t K, int64_t n_in, int64_t n_out, int32_t* imap_t)
{
    for (int64_t j = 0; j < K * n_in; ++j) imap_t[j] = -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t o = 0; o < n_out; ++o) {
            int32_t i = imap[k * n_out + o];
            if (i >= 0) imap_t[k * n_in + i] = (int32_t)o;
        }
}

/* One output row of the forward sum. */
static void fwd_row(const double* x, const double* w, const double* bias, const int32_t* imap,
                    int64_t K, int64_t n_out, int32_t cin, int32_t cout, int64_t o, double* yo)
{
    for (int32_t j = 0; j < cout; ++j) yo[j] = bias ? bias[j] : 0.0;
    for (int64_t k = 0; k < K; ++k) {
        int32_t i = imap[k * n_out + o];
        if (i < 0) continue;
        const double* xi = x + (int64_t)i * cin;
        const double* wk = w + k * cin * cout;
        for (int32_t c = 0; c < cin; ++c)
            for (int32_t j = 0; j < cout; ++j) yo[j] += xi[c] * wk[(int64_t)c * cout + j];
    }
}

void orc_conv_fwd(const double* x, const double* w, const double* bias, const int32_t* imap,
                  int64_t K, int64_t n_in, int64_t n_out, int32_t cin, int32_t cout, double* y)
{
    (void)n_in;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t o = 0; o < n_out; ++o) fwd_row(x, w, bias, imap, K, n_out, cin, cout, o, y + o * cout);
}

/* Forward sum at the listed output rows only; y_rows is [n_rows, cout]. */
void orc_conv_fwd_rows(const double* x, const double* w, const double* bias, const int32_t* imap,
                       int64_t K, int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                       const int64_t* rows, int64_t n_rows, double* y_rows)
{
    (void)n_in;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < n_rows; ++r)
        fwd_row(x, w, bias, imap, K, n_out, cin, cout, rows[r], y_rows + r * cout);
}

void orc_conv_dgrad(const double* dy, const double* w, const int32_t* imap, int64_t K, int64_t n_in,
                    int64_t n_out, int32_t cin, int32_t cout, double* dx)
{
    for (int64_t j = 0; j < n_in * cin; ++j) dx[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double* wk = w + k * cin * cout;
        for (int64_t o = 0; o < n_out; ++o) {
            int32_t i = imap[k * n_out + o];
            if (i < 0) continue;
            const double* g = dy + o * cout;
            double* d = dx + (int64_t)i * cin;
            for (int32_t c = 0; c < cin; ++c) {
                double s = 0.0;
                for (int32_t j = 0; j < cout; ++j) s += wk[(int64_t)c * cout + j] * g[j];
                d[c] += s;
            }
        }
    }
}

/*
 * Inverse conv (spconv SparseInverseConv3d, "spconv.pytorch Core Concepts
 * Definitions" / common usage: the inverse of a strided conv that shares its
 * indice key restores the strided conv's input coordinate set).  For every pair
 * (k, o, i) of the strided conv's map imap [K, n_y] (imap[k, o] = i): the
 * feature y[o] of strided output o goes back to input site i through W[k]:
 *     out[i, :] = bias + sum over pairs with imap[k, o] = i of y[o, :] W[k],
 * W [K, cy, cout].  Written as a scatter over the forward map, so it shares no
 * loop with orc_conv_fwd (which gathers through a map of the output rows).
 */
void orc_conv_inverse(const double* y, const double* w, const double* bias, const int32_t* imap,
                      int64_t K, int64_t n_y, int64_t n_out, int32_t cy, int32_t cout, double* out)
{
    for (int64_t i = 0; i < n_out; ++i)
        for (int32_t j = 0; j < cout; ++j) out[i * cout + j] = bias ? bias[j] : 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double* wk = w + k * cy * cout;
        for (int64_t o = 0; o < n_y; ++o) {
            const int32_t i = imap[k * n_y + o];
            if (i < 0) continue;
            const double* f = y + o * cy;
            double* d = out + (int64_t)i * cout;
            for (int32_t j = 0; j < cout; ++j) {
                double s = 0.0;
                for (int32_t c = 0; c < cy; ++c) s += f[c] * wk[(int64_t)c * cout + j];
                d[j] += s;
            }
        }
    }
}

/*
 * Sparse max pooling (spconv SparseMaxPool3d, "spconv.pytorch Layer APIs
 * Reference": a downsampling layer whose dense version is nn.MaxPool3d), on the
 * strided map of its kernel / stride / padding: for each output row o and
 * channel c, the largest x[i, c] over the pairs imap[k, o] = i, taken over the
 * occupied inputs only (the dense max pool of a grid that holds -infinity at
 * empty cells).  arg[o, c] is the first k (in offset order) that reaches the
 * maximum, 255 for a row without pairs (whose output is 0).
 */
void orc_maxpool_fwd(const double* x, const int32_t* imap, int64_t K, int64_t n_in, int64_t n_out,
                     int32_t c, double* y, uint8_t* arg)
{
    (void)n_in;
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t o = 0; o < n_out; ++o)
        for (int32_t j = 0; j < c; ++j) {
            double best = 0.0;
            int found = -1;
            for (int64_t k = 0; k < K; ++k) {
                const int32_t i = imap[k * n_out + o];
                if (i < 0) continue;
                const double v = x[(int64_t)i * c + j];
                if (found < 0 || v > best) {
                    best = v;
                    found = (int)k;
                }
            }
            y[o * c + j] = found < 0 ? 0.0 : best;
            arg[o * c + j] = (uint8_t)(found < 0 ? 255 : found);
        }
}

/* Its input gradient: dy[o, c] goes to the input row of the pair at arg[o, c]. */
void orc_maxpool_dgrad(const double* dy, const int32_t* imap, const uint8_t* arg, int64_t K,
                       int64_t n_in, int64_t n_out, int32_t c, double* dx)
{
    (void)K;
    for (int64_t j = 0; j < n_in * c; ++j) dx[j] = 0.0;
    for (int64_t o = 0; o < n_out; ++o)
        for (int32_t j = 0; j < c; ++j) {
            const int k = arg[o * c + j];
            if (k == 255) continue;
            const int32_t i = imap[(int64_t)k * n_out + o];
            dx[(int64_t)i * c + j] += dy[o * c + j];
        }
}

/* dinput at the listed input rows, through a transposed map imap_t [K, n_in]. */
void orc_conv_dgrad_rows(const double* dy, const double* w, const int32_t* imap_t, int64_t K,
                         int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                         const int64_t* rows, int64_t n_rows, double* dx_rows)
{
    (void)n_out;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t i = rows[r];
        double* d = dx_rows + r * cin;
        for (int32_t c = 0; c < cin; ++c) d[c] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            int32_t o = imap_t[k * n_in + i];
            if (o < 0) continue;
            const double* wk = w + k * cin * cout;
            const double* g = dy + (int64_t)o * cout;
            for (int32_t c = 0; c < cin; ++c) {
                double s = 0.0;
                for (int32_t j = 0; j < cout; ++j) s += wk[(int64_t)c * cout + j] * g[j];
                d[c] += s;
            }
        }
    }
}

void orc_conv_wgrad(const double* x, const double* dy, const int32_t* imap, int64_t K, int64_t n_in,
                    int64_t n_out, int32_t cin, int32_t cout, double* dw)
{
    (void)n_in;
    for (int64_t j = 0; j < K * cin * cout; ++j) dw[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double* dk = dw + k * cin * cout;
        for (int64_t o = 0; o < n_out; ++o) {
            int32_t i = imap[k * n_out + o];
            if (i < 0) continue;
            const double* xi = x + (int64_t)i * cin;
            const double* g = dy + o * cout;
            for (int32_t c = 0; c < cin; ++c)
                for (int32_t j = 0; j < cout; ++j) dk[(int64_t)c * cout + j] += xi[c] * g[j];
        }
    }
}

/* dfilter at listed flat indices (k * cin + c) * cout + j of dW. */
void orc_conv_wgrad_entries(const double* x, const double* dy, const int32_t* imap, int64_t K,
                            int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                            const int64_t* entries, int64_t n_entries, double* vals)
{
    (void)n_in;
    (void)K;
    for (int64_t e = 0; e < n_entries; ++e) {
        int64_t f = entries[e];
        int64_t j = f % cout, c = (f / cout) % cin, k = f / ((int64_t)cout * cin);
        double s = 0.0;
        for (int64_t o = 0; o < n_out; ++o) {
            int32_t i = imap[k * n_out + o];
            if (i >= 0) s += x[(int64_t)i * cin + c] * dy[o * cout + j];
        }
        vals[e] = s;
    }
}

/*
 * Quantized forward: spconv's int8 implicit GEMM with per-output-channel scale
 * and bias (spconv docs, TENSORRT_INT8_GUIDE.md: "Spconv Int8 Scale/Bias
 * Conversion Basic Rule", "Call Spconv Implicit GEMM with Calculated Scales and
 * Bias", "Calculate Spconv Int8 Scale and Bias from PyTorch Quantized Layer").
 * Values are int8 codes; a code q stands for q * its scale, and a real value v
 * is stored as saturate(round(v / scale)).  With
 *   scale[j] = input_scale * weight_scale[j] / output_scale,
 *   bias[j]  = bias_fp[j] / output_scale,
 * the output code of row o, channel j is
 *   acc = sum over pairs (k, i = imap[k, o] != -1) of sum_c x[i, c] w[k, c, j]
 *         (exact integer sum, kept in 32 bits as the integer GEMM does),
 *   f   = float(acc) * scale[j] + bias[j],
 *   f   = f + add_scale * float(add[o, j])   (fused residual add, when given),
 *   f   = max(f, 0)                          (ReLU, when asked),
 *   y   = saturate(round(f)) to [-128, 127], round half away from zero
 *         (C's round, the plain reading of the rule's round()).
 * Every floating-point operation is an fp32 operation rounded once, in the
 * order written (the rule's data are fp32); nothing is fused.  acc_out
 * (nullable) receives the integer sums.  Returns ORC_ERR_ARG if a sum leaves
 * the 32-bit range.
 */
/* One output row of the int8 rule; returns 1 if a sum leaves the 32-bit range. */
static int fwd_int8_row(const int8_t* x, const int8_t* w, const float* scale, const float* bias,
                        const int8_t* add, float add_scale, int32_t relu, const int32_t* imap,
                        int64_t K, int64_t n_out, int32_t cin, int32_t cout, int64_t o, int64_t* acc,
                        int8_t* yo, int32_t* acc_o)
{
    for (int32_t j = 0; j < cout; ++j) acc[j] = 0;
    for (int64_t k = 0; k < K; ++k) {
        int32_t i = imap ? imap[k * n_out + o] : (int32_t)o;
        if (i < 0) continue;
        const int8_t* xi = x + (int64_t)i * cin;
        const int8_t* wk = w + k * cin * cout;
        for (int32_t c = 0; c < cin; ++c)
            for (int32_t j = 0; j < cout; ++j) acc[j] += (int64_t)xi[c] * (int64_t)wk[(int64_t)c * cout + j];
    }
    for (int32_t j = 0; j < cout; ++j) {
        if (acc[j] > INT32_MAX || acc[j] < INT32_MIN) return 1;
        if (acc_o) acc_o[j] = (int32_t)acc[j];
        float f = (float)(int32_t)acc[j];
        f = f * scale[j];
        if (bias) f = f + bias[j];
        if (add) {
            float t = add_scale * (float)add[o * cout + j];
            f = f + t;
        }
        if (relu && f < 0.0f) f = 0.0f;
        float r = roundf(f);
        if (r > 127.0f) r = 127.0f;
        if (r < -128.0f) r = -128.0f;
        yo[j] = (int8_t)r;
    }
    return 0;
}

int orc_conv_fwd_int8(const int8_t* x, const int8_t* w, const float* scale, const float* bias,
                      const int8_t* add, float add_scale, int32_t relu, const int32_t* imap,
                      int64_t K, int64_t n_in, int64_t n_out, int32_t cin, int32_t cout, int8_t* y,
                      int32_t* acc_out)
{
    (void)n_in;
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        int64_t* acc = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cout > 0 ? cout : 1));
        if (!acc) {
            bad |= 2;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t o = 0; o < n_out; ++o)
                bad |= fwd_int8_row(x, w, scale, bias, add, add_scale, relu, imap, K, n_out, cin,
                                    cout, o, acc, y + o * cout, acc_out ? acc_out + o * cout : NULL);
            free(acc);
        }
    }
    if (bad & 2) return ORC_ERR_NOMEM;
    return bad ? ORC_ERR_ARG : ORC_OK;
}
