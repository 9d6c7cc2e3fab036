// noalloc.cu -- spc_build_indice_map_noalloc: the indice-map build with its hash
// table in a fixed array of device memory owned by the library, for callers
// that cannot allocate device memory themselves.
//
// The table lives in a file-scope __device__ array of SPC_NOALLOC_MAX_VOXELS * 2
// 64-bit slots (16 MiB).  Every device that loads this library holds that
// array until the process exits.  In host code the array's name is only a
// host-side stand-in, never a device address, so the entry point looks the
// real address up once per device with cudaGetSymbolAddress (with that device
// current) and hands that pointer to the kernels as their workspace.
//
// All calls on a device share the one table.  Each call clears it before use,
// so no state carries from one call to the next, but calls whose work overlaps
// on the GPU (different streams, or different host threads) race on it and
// must be serialised by the caller.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr int64_t kMaxVoxels = SPC_NOALLOC_MAX_VOXELS;
constexpr int64_t kSlots = 2 * kMaxVoxels;  // load factor <= 1/2, as for the workspace path

static __device__ __align__(256) unsigned long long g_noalloc_table[kSlots];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_table_addr[kMaxDevices] = {nullptr};

// Device address of the table on the current device (looked up once per device).
spc_status table_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_table_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_table) != cudaSuccess || !p) return SPC_ERR_CUDA;
        g_table_addr[dev] = p;
    }
    *out = g_table_addr[dev];
    return SPC_OK;
}

}  // namespace

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
    const spc_status s = table_address(&table);
    if (s != SPC_OK) return s;
    return spc_build_indice_map(coords, n_in, batch, in_shape, g, subm, out_coords, n_out, imap,
                                imap_t, pair_count, mask, status, table,
                                sizeof(unsigned long long) * (size_t)kSlots, stream);
}
