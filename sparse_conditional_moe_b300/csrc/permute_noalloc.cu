// permute_noalloc.cu -- moe_permute_noalloc: the grouping step (moe_permute) for callers that
// cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the point where they run this step: a plugin
// whose host interface has no workspace argument, or a serving process whose device memory is
// owned entirely by another allocator, where a cudaMalloc in the middle of serving would either
// fail under fragmentation or synchronise the whole device.  For them the two per-block tables
// the grouping kernels need (per-block expert histograms and their running bases) live in a
// fixed array of this library's device image instead of a caller workspace.
//
// Limits and sharing:
//   - The array holds kNoAllocTableEntries int32 per table; a call needs
//     ceil(N*k / 2048) * E entries per table and is rejected with MOE_ERR_WORKSPACE above that.
//   - Every GPU that loads the library keeps this 1 MiB array until the process exits.
//   - All calls on a device share the array, which keeps the last call's contents.  Nothing in
//     it has to start at zero: each call writes every entry it later reads.  Calls whose work
//     overlaps on the GPU (for instance on two streams without ordering) race on the array.
//   - The first call on each device looks up the array's device address (with that device
//     current) and keeps it for the life of the process; make that first call before any stream
//     capture.  A device reset (cudaDeviceReset) after that first call is not supported: the
//     module is loaded again at another address while the kept one goes stale.
#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr int kNoAllocTableEntries = 131072;   // per table: perm blocks x experts
constexpr int kMaxDevices = 64;

// [0, N) per-block histograms, [N, 2N) per-block bases.  In host code this name is only a
// stand-in for the symbol: the kernels get the address looked up below.
static __device__ __align__(256) int32_t g_permute_tables[2 * kNoAllocTableEntries];

std::mutex g_mu;
int32_t* g_tables_addr[kMaxDevices] = {};

// Device address of g_permute_tables on the current device (looked up once per device).
moe_status tables_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_tables_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_tables) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        g_tables_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_tables_addr[dev];
    return MOE_OK;
}

bool ok_ptr(const void* p, size_t align) {
    return p != nullptr && reinterpret_cast<uintptr_t>(p) % align == 0;
}

}  // namespace

extern "C" MOE_API moe_status moe_permute_noalloc(
    const moe_cfg* cfg, const int32_t* idx, const float* w, const void* x, int32_t* counts,
    int32_t* offsets, int32_t* kept, int32_t* kept_offsets, int32_t* perm, int32_t* pos,
    int32_t* row_token, float* row_weight, void* x_perm, int32_t* err, void* stream) {
    size_t unused = 0;
    moe_status st = moe_workspace_size(cfg, &unused);   // validates the configuration
    if (st != MOE_OK) return st;
    if (!ok_ptr(counts, 4) || !ok_ptr(offsets, 4) || !ok_ptr(kept, 4) || !ok_ptr(kept_offsets, 4))
        return MOE_ERR_INVALID_ARG;
    if (cfg->N > 0 &&
        (!ok_ptr(idx, 4) || !ok_ptr(w, 4) || !ok_ptr(x, 16) || !ok_ptr(perm, 4) ||
         !ok_ptr(pos, 4) || !ok_ptr(row_token, 4) || !ok_ptr(row_weight, 4) || !ok_ptr(x_perm, 16)))
        return MOE_ERR_INVALID_ARG;
    if (err != nullptr && !ok_ptr(err, 4)) return MOE_ERR_INVALID_ARG;
    const int64_t entries = (int64_t)moe::perm_blocks(cfg->N * cfg->k) * cfg->E;
    if (entries > kNoAllocTableEntries) return MOE_ERR_WORKSPACE;
    int32_t* tables = nullptr;
    st = tables_for_current_device(&tables);
    if (st != MOE_OK) return st;
    cudaError_t e = moe::launch_permute(*cfg, idx, w, x, counts, offsets, kept, kept_offsets, perm,
                                        pos, row_token, row_weight, x_perm, tables,
                                        tables + kNoAllocTableEntries, err, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
