/*
 * spc.h -- C ABI of libspc.so: sparse 3-D convolution over voxel coordinate sets.
 *
 * The library computes, on one CUDA GPU (sm_103a):
 *   - the indice map (kernel map) of a submanifold or strided sparse conv,
 *     built with a GPU open-addressing hash table over int64 cell keys;
 *   - the output coordinate set of a strided sparse conv (sort + unique);
 *   - the convolution forward, its input gradient (dinput) and its weight
 *     gradient (dfilter) as implicit GEMMs over that map.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Coordinates   int32 [n, 4] row-major rows (b, z, y, x), batch index first
 *                (spconv docs, USAGE.md "Core Concepts Definitions": the
 *                indices of a sparse conv tensor are stored transposed, one row
 *                per voxel).  The pointer must be 16-byte aligned.
 *  Grid          in_shape = (D, H, W) of the (z, y, x) axes, batch in [0, batch).
 *  Kernel index  k runs in C order over (kz, ky, kx); K = kz*ky*kx (lato_mlx
 *                sparse/conv.py, "_kernel_offsets": centred offsets in C order
 *                over (dz, dy, dx), the ordering spconv uses).
 *  Weights       [K, Cin, Cout] row-major (lato_mlx sparse/conv.py, SubMConv3d
 *                class docstring, weight layout).
 *  Features      [rows, C] row-major; dtype given by spc_dtype.
 *  Indice map    int32 [K, n_out] row-major: imap[k, o] is the input row that
 *                output row o reads through offset k, or -1 when that cell is
 *                empty or outside the grid.
 *  Pointers      every array argument is a DEVICE pointer owned by the caller,
 *                except those marked "host".  The library keeps no state and
 *                allocates nothing: scratch memory is a caller-supplied
 *                workspace of at least the size the matching *_workspace_size
 *                query returns (256-byte aligned).
 *  Streams       `stream` is a cudaStream_t (NULL = legacy default stream);
 *                all device work is enqueued on it and no call synchronises.
 *  Errors        Argument errors are returned synchronously, before any work
 *                is enqueued.  Errors that depend on the data (a coordinate out
 *                of range, a duplicate coordinate, a full hash table, an output
 *                set larger than its buffer) are written to `status`, a device
 *                int32 the caller zeroes once: a kernel that finds an error
 *                stores its spc_status there only if it still holds SPC_OK, so
 *                the first error sticks.  Read it after synchronising.
 *                Results written alongside a nonzero status are unspecified.
 *  Empty input   n = 0 (or an empty output set) is valid and does no work.
 */
#ifndef SPC_H
#define SPC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPC_API __attribute__((visibility("default")))
#else
#define SPC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPC_OK = 0,
    SPC_ERR_INVALID_ARG = 1,   /* bad size, null pointer, misaligned pointer, bad geometry */
    SPC_ERR_COORD_RANGE = 2,   /* a coordinate lies outside [0,batch) x grid */
    SPC_ERR_DUPLICATE = 3,     /* two rows hold the same (b, z, y, x) */
    SPC_ERR_TABLE_FULL = 4,    /* a hash probe exceeded its bound */
    SPC_ERR_CAPACITY = 5,      /* the strided output set exceeds the caller's buffer */
    SPC_ERR_UNSUPPORTED = 6,   /* a valid request this build does not implement */
    SPC_ERR_CUDA = 7,          /* a CUDA runtime call failed (launch, copy) */
    SPC_ERR_WORKSPACE = 8,     /* workspace missing or smaller than required */
    SPC_ERR_TIMEOUT = 9        /* an internal GPU wait exceeded its bound (spc_set_wait_limit_ns); results invalid */
} spc_status;

typedef enum { SPC_F32 = 0, SPC_F16 = 1, SPC_BF16 = 2 } spc_dtype;

/* SPC_PREC_EXACT: fp32 features use full fp32 multiplies; fp16/bf16 features
 * multiply exactly (their products fit fp32) and accumulate in fp32.
 * SPC_PREC_TF32: fp32 features are rounded to tf32 before a tensor-core
 * multiply (accumulation stays fp32); ignored for fp16/bf16. */
typedef enum { SPC_PREC_EXACT = 0, SPC_PREC_TF32 = 1 } spc_precision;

/* Activation of the fused forward epilogue (spc_conv_fwd_fused). */
typedef enum { SPC_ACT_NONE = 0, SPC_ACT_RELU = 1 } spc_activation;

/* How spc_conv_dgrad reads its map argument. */
typedef enum {
    /* map is the transposed map imap_t [K, n_in]: imap_t[k, i] = o for every
     * pair imap[k, o] = i (what spc_build_indice_map writes for strided maps). */
    SPC_MAP_TRANSPOSED = 0,
    /* map is a submanifold map imap [K, n] (n_in == n_out): its transpose is
     * its offset mirror, imap_t[k, i] = imap[K-1-k, i], so no second map is kept. */
    SPC_MAP_SUBM_MIRROR = 1
} spc_map_kind;

/* Convolution geometry per axis (z, y, x). */
typedef struct {
    int32_t ksize[3];
    int32_t stride[3];
    int32_t pad[3];
    int32_t dil[3];
} spc_geom;

/* Human-readable name of a status code (static storage). */
SPC_API const char* spc_status_string(spc_status s);

/* Library version as major*10000 + minor*100 + patch. */
SPC_API int32_t spc_version(void);

/* Bound on the waits inside the pipelined tensor-core kernels (conv forward,
 * dinput, inverse, dfilter) of one warp role on another: a gather warp waiting
 * for a free stage, the MMA thread waiting for a full one.  Such a wait never
 * lasts long in a healthy run; one that runs out makes the kernel set
 * SPC_ERR_TIMEOUT in the call's status word, wait for the copies and MMAs it
 * issued itself (those always finish; bounded by 2 s), free its tensor memory
 * and return, so the context stays usable.  The limit applies to kernels
 * launched (or captured into a graph) after the call; process-wide; default
 * 2,000,000,000 ns, at most 60 s (SPC_ERR_INVALID_ARG above).  A limit of 0
 * gives up at the first such wait whose phase is not already complete.  The
 * limit is checked between suspended polls of up to 100 us, so a wait may run
 * past it by that much. */
SPC_API spc_status spc_set_wait_limit_ns(uint64_t ns);
SPC_API uint64_t spc_get_wait_limit_ns(void);

/* Output grid of a strided (regular) sparse conv, per axis
 * floor((in + 2 pad - dil (k - 1) - 1) / stride) + 1, or 0 when the window never
 * fits: the grid a dense conv over the densified input produces (spconv docs,
 * USAGE.md "Core Concepts Definitions", Sparse Convolution).  Host only. */
SPC_API spc_status spc_out_shape(const int32_t in_shape[3] /*host*/, const spc_geom* g /*host*/,
                         int32_t out_shape[3] /*host, out*/);

/* ------------------------------------------------------------------ indice map
 * spc_build_indice_map -- validate and key the input coordinates, build the
 * hash table, and probe every (output row, offset) pair.
 *
 *  subm != 0 (submanifold conv; spconv USAGE.md "Core Concepts Definitions",
 *    Submanifold Convolution; lato_mlx sparse/conv.py "build_indice_map"):
 *    the output set is the input set (out_coords ignored, n_out must equal
 *    n_in), every ksize must be odd, stride and pad are ignored, and offset k
 *    reads the cell coords[o] + ((kz - ksz/2) dil_z, (ky - ksy/2) dil_y,
 *    (kx - ksx/2) dil_x).
 *  subm == 0 (strided conv): output row o = out_coords[o] (grid
 *    spc_out_shape(in_shape, g)) reads input cell out*stride - pad + k*dil.
 *
 *  coords     [n_in, 4] int32 input coordinates (16-byte aligned).
 *  out_coords [n_out, 4] int32 output coordinates (strided only, else NULL).
 *  imap       [K, n_out] int32 out: input row or -1.
 *  imap_t     [K, n_in] int32 out or NULL: output row or -1, the transpose of
 *             imap (strided only; must be NULL when subm != 0).
 *  pair_count [K] int32 out: number of entries != -1 in each row of imap.
 *  mask       [n_out] uint32 out or NULL: bit k set when imap[k, o] != -1
 *             (only when K <= 32).
 *  status     device int32, sticky error word (see above).  Sets
 *             SPC_ERR_COORD_RANGE, SPC_ERR_DUPLICATE or SPC_ERR_TABLE_FULL.
 *  ws         workspace of spc_indice_map_workspace_size(n_in) bytes.
 */
SPC_API size_t spc_indice_map_workspace_size(int64_t n_in);

SPC_API spc_status spc_build_indice_map(const int32_t* coords, int64_t n_in, int32_t batch,
                                const int32_t in_shape[3] /*host*/, const spc_geom* g /*host*/,
                                int32_t subm, const int32_t* out_coords, int64_t n_out,
                                int32_t* imap, int32_t* imap_t, int32_t* pair_count,
                                uint32_t* mask, int32_t* status, void* ws, size_t ws_bytes,
                                void* stream);

/* spc_build_indice_map_noalloc -- the same indice-map build as
 * spc_build_indice_map, for callers that cannot allocate device memory: an
 * inference engine's enqueue step that must not call cudaMalloc/cudaFree
 * (they can stall the whole device), a host framework that owns all device
 * memory through its own pool and offers no workspace, or a latency-bound loop
 * that sized every buffer at start-up.  The pages describe no such variant;
 * it has no counterpart there.
 *
 *  Arguments are those of spc_build_indice_map without ws / ws_bytes; the hash
 *  table lives instead in a 16 MiB array of device memory inside the library,
 *  which every GPU that loads the library keeps until the process exits.
 *  n_in may be at most SPC_NOALLOC_MAX_VOXELS; larger inputs return
 *  SPC_ERR_WORKSPACE before any work is enqueued.
 *  The first call in a CUDA context looks up the array's device address in
 *  that context (with the caller's device current) and caches it by the
 *  context's unique id; after cudaDeviceReset or in another context the
 *  array sits at another address, and the next call there looks it up again.
 *  Make the first call in a context before any stream capture.  The call
 *  allocates nothing and synchronises nothing.
 *  All calls in a context share the one table.  Each call clears it before use,
 *  but calls whose GPU work overlaps (other streams, other host threads) race
 *  on it: the caller must serialise them. */
#define SPC_NOALLOC_MAX_VOXELS 1048576

SPC_API spc_status spc_build_indice_map_noalloc(const int32_t* coords, int64_t n_in,
                                                int32_t batch, const int32_t in_shape[3] /*host*/,
                                                const spc_geom* g /*host*/, int32_t subm,
                                                const int32_t* out_coords, int64_t n_out,
                                                int32_t* imap, int32_t* imap_t,
                                                int32_t* pair_count, uint32_t* mask,
                                                int32_t* status, void* stream);

/* ------------------------------------------------------ strided output coords
 * spc_strided_out_coords -- output coordinate set of a strided sparse conv:
 * every cell of the output grid whose receptive field (out*stride - pad +
 * k*dil over all k) holds at least one input voxel of the same batch.  Output
 * cells outside the output grid do not exist, so inputs that reach none are
 * dropped (spconv docs, COMMON_PROBLEMS.md: shape [8,200,200], k3 s2 pad
 * [0,1,1], the single point z=7 gives an empty output).  Rows are written
 * sorted by (b, z, y, x).
 *
 *  out_shape   host out: the output grid (as spc_out_shape).
 *  out_coords  [cap, 4] int32 out (16-byte aligned).
 *  n_out       device int64 out: size of the output set, written even when it
 *              exceeds cap (then SPC_ERR_CAPACITY is set in status and
 *              out_coords holds only a prefix).
 *  status      sticky error word: SPC_ERR_COORD_RANGE, SPC_ERR_CAPACITY.
 *  ws          spc_strided_out_coords_workspace_size(n_in, g) bytes.
 *  The caller reads n_out back to size the following buffers; cap = n_in * K
 *  always suffices.
 */
SPC_API size_t spc_strided_out_coords_workspace_size(int64_t n_in, const spc_geom* g /*host*/);

SPC_API spc_status spc_strided_out_coords(const int32_t* coords, int64_t n_in, int32_t batch,
                                  const int32_t in_shape[3] /*host*/, const spc_geom* g /*host*/,
                                  int32_t out_shape[3] /*host, out*/, int32_t* out_coords,
                                  int64_t cap, int64_t* n_out, int32_t* status, void* ws,
                                  size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------- conv
 * spc_conv_fwd -- y[o, :] = bias + sum_k sum_{i = imap[k, o] != -1} x[i, :] W[k]
 * (lato_mlx sparse/conv.py, module docstring: the output is the bias plus, over
 * the kernel offsets, the weight slice times the feature of each occupied
 * neighbour; absent neighbours add nothing).  One launch covers all offsets;
 * each output row is written once (no atomics: results are run-to-run
 * bit-identical).
 *
 *  x     [n_in, cin] of dtype dt.      w [K, cin, cout] of dtype dt.
 *  bias  [cout] of dtype dt, or NULL.
 *  imap  [K, n_out] int32, or NULL when K == 1 and n_in == n_out: the 1x1
 *        submanifold conv is a per-voxel linear layer y = x W[0] + bias and
 *        needs no map (lato_mlx sparse/conv.py, SubMConv3d.__call__ k=1
 *        shortcut; HYGON-AI spconv-das README, 1x1 takes the GEMM path).
 *  mask  [n_out] uint32 or NULL: the per-row offset mask from
 *        spc_build_indice_map; the narrow-channel kernel walks only a row's
 *        set bits (the tensor-core kernel reads all of a row's map entries in
 *        one burst and skips the offsets no row of its tile uses).
 *  y     [n_out, cout] of dtype dt out (fp32 accumulate, one rounding).
 *  status  device int32 sticky error word, or NULL (SPC_ERR_TIMEOUT).
 *  ws    spc_conv_workspace_size(...) bytes: 0 when the tensor-core path reads
 *        W as stored (fp16 / bf16 with Cin and Cout multiples of 64); the
 *        other tensor-core shapes keep the weights transposed to [K, Cout, Cin]
 *        there.
 *  x, w, y must be 16-byte aligned.
 *  Kernels: a one-row-per-thread kernel when Cin and Cout are both in
 *  {8, 16, 32} (narrow layers on sparse scenes are latency-bound); else
 *  tcgen05 tensor cores when the channels allow (fp16 / bf16 with Cin % 64 ==
 *  0, or 16 / 32 with Cout % 64 == 0, or fp32 with SPC_PREC_TF32 and Cin % 32
 *  == 0; Cout % 64 == 0 or in {16, 32}; K <= 32); else a tiled CUDA-core kernel.
 */
SPC_API size_t spc_conv_workspace_size(int32_t K, int64_t n_in, int64_t n_out, int32_t cin,
                               int32_t cout, spc_dtype dt);

SPC_API spc_status spc_conv_fwd(const void* x, const void* w, const void* bias,
                                const int32_t* imap, const uint32_t* mask, int32_t K,
                                int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                                spc_dtype dt, spc_precision prec, void* y, int32_t* status,
                                void* ws, size_t ws_bytes, void* stream);

/* spc_conv_fwd_fused -- y[o, :] = act(bias + sum_k sum_{i = imap[k, o] != -1} x[i, :] W[k]
 *                                     + add_scale * residual[o, :])
 * (spconv docs, "Call Spconv Implicit GEMM with Calculated Scales and Bias":
 * the implicit GEMM takes a bias, an activation and an added output with its
 * scale, "for fused conv-add-relu layer"; "Fusible Spconv Residual Block
 * Example for Quantization": out = relu(conv_bn(x) + identity)).  The residual
 * add and the activation run in the forward's epilogue on the fp32
 * accumulators, before the single rounding to dt, so the output is written in
 * one pass and the residual read once.
 *
 *  perm       [n_out] int32 or NULL: a row order from spc_map_row_order(imap)
 *             (rows grouped by offset mask; pass its mask as `mask`).  The
 *             tensor-core kernel then computes its row tiles in that order and
 *             a tile runs only the offsets its rows use: on submanifold shells
 *             that cuts the tiles' zero-filled rows from about a fifth of the
 *             gathered slots to a few percent (spconv's mask-sorted implicit
 *             GEMM, the `do_sort` of "Optimize Int8 Kernels by Disabling Sort
 *             in Implicit Gemm").  The result is the same; K <= 32.
 *  residual   [n_out, cout] of dtype dt, 16-byte aligned, or NULL (no add);
 *             it must not be y itself.
 *  add_scale  factor of the residual (1.0 for a plain residual add).
 *  act        SPC_ACT_NONE or SPC_ACT_RELU.
 *  All other arguments, the kernels and the errors as for spc_conv_fwd, which is
 *  this call with perm and residual NULL and SPC_ACT_NONE.
 */
SPC_API spc_status spc_conv_fwd_fused(const void* x, const void* w, const void* bias,
                                      const int32_t* imap, const uint32_t* mask,
                                      const int32_t* perm, int32_t K, int64_t n_in, int64_t n_out,
                                      int32_t cin, int32_t cout, spc_dtype dt, spc_precision prec,
                                      const void* residual, float add_scale, spc_activation act,
                                      void* y, int32_t* status, void* ws, size_t ws_bytes,
                                      void* stream);

/* spc_conv_inverse -- out[i, :] = bias + sum over pairs imap[k, o] = i of y[o, :] W[k]
 * (spconv SparseInverseConv3d, "spconv.pytorch Layer APIs Reference" and "Using
 * SparseInverseConv for Inverse Sparse Operations": the inverse of a strided
 * conv that shares its indice key; it brings features on the strided conv's
 * output set back to that conv's input set through the same pairs).  Read
 * through the strided conv's transposed map, it is a gathered conv like
 * spc_conv_fwd with the roles of the two coordinate sets exchanged, and runs on
 * the same kernels.  Its gradients are spc_conv_dgrad with the forward map imap
 * as SPC_MAP_TRANSPOSED (dy = sum over pairs of W[k] dout[i]) and
 * spc_conv_wgrad(y, dout, imap_t) (dW[k] = sum over pairs of y[o]^T dout[i]).
 *
 *  y      [n_y, cy] of dtype dt: features on the strided conv's output set.
 *  w      [K, cy, cout] of dtype dt.   bias [cout] or NULL.
 *  imap_t [K, n_out] int32: the strided conv's transposed map from
 *         spc_build_indice_map (imap_t[k, i] = o exactly when imap[k, o] = i).
 *  mask_t, perm  [n_out] uint32 / int32 from spc_map_row_order(imap_t), or
 *         NULL (K <= 32 when given).  With them the tensor-core kernel computes
 *         its row tiles in an order that groups rows using the same offsets,
 *         and a tile runs only those offsets; the result is the same.
 *  out    [n_out, cout] of dtype dt out: rows of the strided conv's input set.
 *  ws     spc_conv_workspace_size(K, n_y, n_out, cy, cout, dt) bytes.
 *  Errors and alignment as for spc_conv_fwd.
 */
SPC_API spc_status spc_conv_inverse(const void* y, const void* w, const void* bias,
                                    const int32_t* imap_t, const uint32_t* mask_t,
                                    const int32_t* perm, int32_t K, int64_t n_y, int64_t n_out,
                                    int32_t cy, int32_t cout, spc_dtype dt, spc_precision prec,
                                    void* out, int32_t* status, void* ws, size_t ws_bytes,
                                    void* stream);

/* spc_conv_fwd_int8 -- quantized forward, spconv's int8 implicit GEMM (spconv
 * docs, TENSORRT_INT8_GUIDE.md: "Spconv Int8 Scale/Bias Conversion Basic Rule",
 * fp32 = int8 * scale and int8 = saturate(round(fp32 / scale)); "Call Spconv
 * Implicit GEMM with Calculated Scales and Bias"; "Calculate Spconv Int8 Scale
 * and Bias from PyTorch Quantized Layer", scale = input_scale *
 * weight_scale[j] / output_scale and bias = bias_fp / output_scale):
 *   acc[o, j] = sum over pairs (k, i = imap[k, o] != -1) of sum_c x[i, c] w[k, c, j]
 *               (exact integer sum),
 *   f = float(acc) * scale[j] + bias[j] + add_scale * float(add[o, j]),
 *   f = max(f, 0) with SPC_ACT_RELU,
 *   y[o, j] = saturate(round(f)) to [-128, 127], round half away from zero;
 * each fp32 operation rounded once in that order (nothing fused), so the codes
 * are bit-exact against a CPU evaluation of the same expression.
 * sm_103a has no integer tensor-core MMA; the sums are formed exactly on the
 * fp16 tensor cores (int8 values are exact in fp16; each weight is split into
 * two 4-bit halves so every fp32 partial sum is an exact integer), which needs
 * K * cin <= 8192.
 *
 *  x      [n_in, cin] int8.   w [K, cin, cout] int8.
 *  scale  [cout] fp32 (device).   bias [cout] fp32 (device) or NULL.
 *  imap   [K, n_out] int32, or NULL when K == 1 and n_in == n_out.
 *  mask, perm  [n_out] uint32 / int32 from spc_map_row_order(imap), or NULL:
 *         with them tiles of rows grouped by offset mask run only their
 *         offsets (spconv's do_sort); NULL keeps rows in map order (do_sort =
 *         false, "Optimize Int8 Kernels by Disabling Sort in Implicit Gemm").
 *         The result is the same either way.
 *  add    [n_out, cout] int8 residual (16-byte aligned, not y) or NULL;
 *         add_scale its fp32 scale relative to the output.
 *  act    SPC_ACT_NONE or SPC_ACT_RELU.
 *  y      [n_out, cout] int8 out.
 *  status device int32 sticky error word, or NULL (SPC_ERR_TIMEOUT).
 *  ws     spc_conv_int8_workspace_size(K, cin, cout) bytes, 256-byte aligned
 *         (the split weights, fp16 [K, 2 cout, cin]).
 *  x, w, y must be 16-byte aligned.  cin and cout multiples of 64, K <= 32 and
 *  K * cin <= 8192, else SPC_ERR_UNSUPPORTED (the workspace size is then 0).
 */
SPC_API size_t spc_conv_int8_workspace_size(int32_t K, int32_t cin, int32_t cout);
SPC_API spc_status spc_conv_fwd_int8(const int8_t* x, const int8_t* w, const float* scale,
                                     const float* bias, const int32_t* imap, const uint32_t* mask,
                                     const int32_t* perm, int32_t K, int64_t n_in, int64_t n_out,
                                     int32_t cin, int32_t cout, const int8_t* add, float add_scale,
                                     spc_activation act, int8_t* y, int32_t* status, void* ws,
                                     size_t ws_bytes, void* stream);

/* spc_map_row_order -- the rows of a map [K, n] grouped by offset mask.
 * mask[i] gets bit k when map[k, i] != -1, and perm lists the rows sorted by
 * mask (stable: rows keep their order within a group).  For the transposed map
 * of a strided conv the groups are the stride's residue classes of the input
 * coordinates, each using only a few offsets, so a tile of grouped rows skips
 * most of the K offsets that a tile of consecutive rows would run (no
 * counterpart on the pages: it is how this library feeds spc_conv_inverse).
 * Computed once per map, like the map itself.  A caller can also permute the
 * voxel rows themselves (coordinates and features) into this order once per
 * indice key and build the map for that order: the convs then need no perm
 * and their tiles still run few zero-filled rows (4 x 192^3 shells, bf16
 * 64 -> 64 forward: 210 us against 241 us in (b, z, y, x) order).
 *
 *  map   [K, n] int32, K <= 32, and mask [n] uint32 out (or NULL); or map NULL
 *        and mask [n] in: the row masks spc_build_indice_map already wrote for
 *        that map (the K x n map is then not read).
 *  perm  [n] int32 out: a permutation of 0 .. n-1.
 *  ws    spc_map_row_order_workspace_size(n) bytes.
 */
SPC_API size_t spc_map_row_order_workspace_size(int64_t n);
SPC_API spc_status spc_map_row_order(const int32_t* map, int32_t K, int64_t n, uint32_t* mask,
                                     int32_t* perm, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ pooling
 * spc_maxpool_fwd -- y[o, c] = max over the pairs imap[k, o] = i of x[i, c]
 * (spconv SparseMaxPool3d, "spconv.pytorch Layer APIs Reference": downsampling
 * whose dense version is nn.MaxPool3d).  The maximum is over the occupied
 * inputs of o's window only, i.e. the dense max pool of a grid holding
 * -infinity at empty cells; on the output set of a strided map every row has
 * at least one pair.  imap is the strided map of the pool's kernel, stride and
 * padding from spc_build_indice_map (subm = 0).
 *
 *  x     [n_in, c] of dtype dt.   y [n_out, c] of dtype dt out (exact: a max).
 *  imap  [K, n_out] int32.        mask [n_out] uint32 or NULL (lets rows skip
 *        offsets without a pair).
 *  arg   [n_out, c] uint8 out or NULL: the first offset k (in offset order)
 *        reaching the maximum, 255 for a row without pairs (whose y is 0);
 *        needed by spc_maxpool_dgrad.
 *  K <= 254 (K <= 32 with a mask); x, y 16-byte aligned for vector access.
 */
SPC_API spc_status spc_maxpool_fwd(const void* x, const int32_t* imap, const uint32_t* mask,
                                   int32_t K, int64_t n_in, int64_t n_out, int32_t c,
                                   spc_dtype dt, void* y, uint8_t* arg, void* stream);

/* spc_maxpool_dgrad -- dx[i, c] = sum over the pairs imap[k, o] = i with
 * arg[o, c] == k of dy[o, c] (the gradient of spc_maxpool_fwd: each output
 * channel passes its gradient to the input it took).  Read through the
 * transposed map, one write per row of dx, no atomics.
 *
 *  dy     [n_out, c] of dtype dt.   imap_t [K, n_in] int32 (the pool map's
 *         transpose, spc_build_indice_map with imap_t).   arg from
 *         spc_maxpool_fwd.   dx [n_in, c] of dtype dt out.
 */
SPC_API spc_status spc_maxpool_dgrad(const void* dy, const int32_t* imap_t, const uint8_t* arg,
                                     int32_t K, int64_t n_in, int64_t n_out, int32_t c,
                                     spc_dtype dt, void* dx, void* stream);

/* spc_conv_dgrad -- dx[i, :] = sum over pairs imap[k, o] = i of W[k] dy[o, :]
 * (the gradient of spc_conv_fwd with respect to x; "dinput" in the HYGON-AI
 * spconv-das README, Testing and Accuracy).  Computed input-stationary through
 * the transposed map, one write per row of dx, no atomics.
 *
 *  dy    [n_out, cout] of dtype dt.   w [K, cin, cout].
 *  map   see spc_map_kind: imap_t [K, n_in] (SPC_MAP_TRANSPOSED) or the
 *        submanifold imap [K, n] (SPC_MAP_SUBM_MIRROR, n_in == n_out); NULL
 *        when K == 1 and n_in == n_out (dx = dy W[0]^T).
 *  mask  NULL, or (K <= 32) with SPC_MAP_SUBM_MIRROR the row mask that
 *        spc_build_indice_map (or spc_map_row_order) wrote for that submanifold
 *        map (the kernel mirrors its bits itself), with SPC_MAP_TRANSPOSED the
 *        mask spc_map_row_order wrote for imap_t.
 *  perm  [n_in] int32 or NULL: a row order of the input rows (for a
 *        submanifold map, the forward's spc_map_row_order(imap) order serves:
 *        mirrored masks group the same way), as for spc_conv_fwd_fused.
 *  dx    [n_in, cin] of dtype dt out.
 *  status  device int32 sticky error word, or NULL (SPC_ERR_TIMEOUT).
 *  Kernels as for spc_conv_fwd with the roles of Cin and Cout exchanged; no
 *  workspace is needed.
 */
SPC_API spc_status spc_conv_dgrad(const void* dy, const void* w, const int32_t* map,
                                  spc_map_kind kind, const uint32_t* mask, const int32_t* perm,
                                  int32_t K, int64_t n_in, int64_t n_out, int32_t cin,
                                  int32_t cout, spc_dtype dt, spc_precision prec, void* dx,
                                  int32_t* status, void* ws, size_t ws_bytes, void* stream);

/* spc_conv_wgrad -- dW[k] = sum_{o: imap[k, o] = i != -1} x[i, :]^T dy[o, :],
 * reduced in fp32 over all active pairs ("dfilter" in the HYGON-AI spconv-das
 * README).  Split over fixed chunks of output rows and summed in a fixed
 * order, so the result is run-to-run bit-identical.
 *
 *  x   [n_in, cin], dy [n_out, cout] of dtype dt;  imap [K, n_out] (NULL when
 *      K == 1 and n_in == n_out).
 *  dw  [K, cin, cout] float32 out (overwritten, not accumulated).
 *  status  device int32 sticky error word, or NULL (SPC_ERR_TIMEOUT).
 *  ws  spc_conv_wgrad_workspace_size(...) bytes (16-byte aligned).
 *  Kernels: tcgen05 tensor cores for fp16 / bf16 with Cin and Cout multiples
 *  of 64 (each CTA: up to 8 offsets, in pairs that share one M = 128 MMA, x a
 *  64 x 64 tile x a fixed row range, accumulators in tensor memory, two CTAs per
 *  SM), else a tiled CUDA-core kernel; partial tiles are then summed over the
 *  row ranges in a fixed order.
 */
SPC_API size_t spc_conv_wgrad_workspace_size(int32_t K, int64_t n_in, int64_t n_out, int32_t cin,
                                     int32_t cout, spc_dtype dt);

SPC_API spc_status spc_conv_wgrad(const void* x, const void* dy, const int32_t* imap, int32_t K,
                                  int64_t n_in, int64_t n_out, int32_t cin, int32_t cout,
                                  spc_dtype dt, spc_precision prec, float* dw, int32_t* status,
                                  void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPC_H */
