// e0_moe_block_forward_noalloc: the decode MoE block for callers that cannot
// provide a workspace.  Its scratch lives in a fixed device array owned by the
// library, so the call allocates nothing and takes no workspace argument.
#include <cuda_runtime.h>

#include <mutex>

#include "e0_common.cuh"
#include "e0_internal.h"

namespace {

// Scratch shared by every call on a device.  Every GPU that loads the library
// holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)E0_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The device address of the scratch array for the current device, looked up
// once per device (with that device current) and cached.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return E0_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return E0_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return E0_OK;
}

}  // namespace

extern "C" int e0_moe_block_forward_noalloc(const float* x, int T, const e0_slot_pool* pool, const uint16_t* W_router,
                                            const e0_route_params* rp, const int32_t* inds_in, const float* w_in,
                                            const e0_shared_expert* shared, float* y, int32_t* inds_out,
                                            float* w_out, uint32_t* d_status, e0_stream_t stream) {
    if (!pool || !rp) return E0_ERR_NULL;
    if (T < 0) return E0_ERR_ARG;
    if (T == 0) return E0_OK;
    const size_t need = e0_workspace_size(0, T, pool->H, pool->I, pool->E, rp->K);
    if (need == 0) return E0_ERR_ARG;
    if (need > kNoAllocScratchBytes) return E0_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != E0_OK) return rc;
    // Nothing in the scratch has to start at zero: every buffer the block
    // uses there is written before it is read within the same call.
    return e0_moe_block_forward(x, T, pool, W_router, rp, inds_in, w_in, shared, y, inds_out, w_out, scratch, need,
                                d_status, stream);
}
