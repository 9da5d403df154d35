// moe_build_slot_map_noalloc: the routing-map stage for callers that cannot
// allocate device memory, so cannot hand the library a workspace.  The stage's
// scratch (device error word and per-chunk expert counts) lives in a
// file-scope device array instead; everything else is the workspace form's
// code path (launch_build_slot_map).
#include <mutex>

#include "common.cuh"

namespace moe {
int launch_build_slot_map(const int32_t*, int, int, int, int32_t*, int32_t*, int32_t*, int32_t*,
                          int32_t*, uint8_t*, cudaStream_t);
}  // namespace moe

using namespace moe;

namespace {

// 256-byte header (error word, counters) + 1 MiB of chunk counts: every GPU
// that loads the library holds these bytes until the process exits.
constexpr size_t kStaticScratchBytes = 256 + (size_t(1) << 20);
__device__ __align__(256) uint8_t g_slot_map_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_slot_map_scratch on the current device, looked up once
// per device (host code only sees a host-side stand-in for the symbol).
int scratch_for_current_device(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_slot_map_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_scratch_ptr[dev]);
    return MOE_OK;
}

}  // namespace

extern "C" int moe_build_slot_map_noalloc(const int32_t* ids, int T, int K, int E,
                                          int32_t* offsets, int32_t* slot, int32_t* src,
                                          int32_t* active, int32_t* n_active, void* stream) {
    if (T < 0 || K < 0 || E <= 0 || E > MAX_E) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (!offsets || !active || !n_active) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K > 0 && (!ids || !slot || !src)) return MOE_ERR_INVALID_ARG;
    // the stage uses the header and the chunk-count table of the workspace layout
    const WsLayout W = ws_layout(T, K, E, 0, 0);
    if (W.chunk_counts + (size_t)W.n_chunks * (size_t)E * sizeof(int32_t) > kStaticScratchBytes)
        return MOE_ERR_UNSUPPORTED;
    uint8_t* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != MOE_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: start from a clear header
    if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_build_slot_map(ids, T, K, E, offsets, slot, src, active, n_active, scratch, s);
}
