// noalloc.cu -- spc_build_indice_map_noalloc: the indice-map build with its hash
// table in a fixed array of device memory owned by the library, for callers
// that cannot allocate device memory themselves.
//
// The table lives in a file-scope __device__ array of SPC_NOALLOC_MAX_VOXELS * 2
// 64-bit slots (16 MiB).  Every device that loads this library holds that
// array until the process exits.  In host code the array's name is only a
// host-side stand-in, never a device address, so the entry point looks the
// real address up with cudaGetSymbolAddress (with the caller's device current)
// and hands that pointer to the kernels as their workspace.
//
// The address belongs to the CUDA context the module was loaded into, not to
// the device number: after cudaDeviceReset, or in another context on the same
// device, the module is loaded again at another address.  The cache is
// therefore keyed by the unique id of the current context (cuCtxGetCurrent and
// cuCtxGetId, reached through the runtime's driver entry points so that nothing
// links libcuda), and a call in a context it has not seen looks the address up
// again.
//
// All calls in a context share the one table.  Each call clears it before use,
// so no state carries from one call to the next, but calls whose work overlaps
// on the GPU (different streams, or different host threads) race on it and
// must be serialised by the caller.
#include "ctx_cache.h"
#include "kernels.cuh"

namespace {

constexpr int64_t kMaxVoxels = SPC_NOALLOC_MAX_VOXELS;
constexpr int64_t kSlots = 2 * kMaxVoxels;  // load factor <= 1/2, as for the workspace path

static __device__ __align__(256) unsigned long long g_noalloc_table[kSlots];

typedef int (*CtxGetCurrentFn)(void**);
typedef int (*CtxGetIdFn)(void*, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name)
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint(name, &p, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Unique id of the current context; false when there is none.
bool current_ctx_id(unsigned long long* id)
{
    static CtxGetCurrentFn get = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    void* ctx = nullptr;
    return get && get_id && get(&ctx) == 0 && ctx && get_id(ctx, id) == 0;
}

spc::CtxCache<16> g_cache;

bool lookup(void** p) { return cudaGetSymbolAddress(p, g_noalloc_table) == cudaSuccess; }

}  // namespace

namespace spc {

// Device address of the table in the caller's current context.
spc_status noalloc_table_address(void** out)
{
    unsigned long long id = 0;
    if (!current_ctx_id(&id)) {
        // no current context yet: the runtime makes the device's primary
        // context current on its first call that needs one
        void* p = nullptr;
        if (!lookup(&p) || !p || !current_ctx_id(&id)) return SPC_ERR_CUDA;
    }
    void* p = g_cache.get(id, lookup);
    if (!p) return SPC_ERR_CUDA;
    *out = p;
    return SPC_OK;
}

}  // namespace spc

extern "C" SPC_API spc_status spc_build_indice_map_noalloc(
    const int32_t* coords, int64_t n_in, int32_t batch, const int32_t in_shape[3],
    const spc_geom* g, int32_t subm, const int32_t* out_coords, int64_t n_out, int32_t* imap,
    int32_t* imap_t, int32_t* pair_count, uint32_t* mask, int32_t* status, void* stream)
{
    if (n_in < 0) return SPC_ERR_INVALID_ARG;
    if (n_in > kMaxVoxels) return SPC_ERR_WORKSPACE;
    const size_t need = spc_indice_map_workspace_size(n_in);
    if (need > sizeof(unsigned long long) * (size_t)kSlots) return SPC_ERR_WORKSPACE;
    void* table = nullptr;
    const spc_status s = spc::noalloc_table_address(&table);
    if (s != SPC_OK) return s;
    return spc_build_indice_map(coords, n_in, batch, in_shape, g, subm, out_coords, n_out, imap,
                                imap_t, pair_count, mask, status, table,
                                sizeof(unsigned long long) * (size_t)kSlots, stream);
}
