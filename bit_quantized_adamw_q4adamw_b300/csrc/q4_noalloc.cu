// q4adamw_step_noalloc: the fused step with its scratch in a fixed, statically
// allocated device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand the library a workspace.  Some run
// inside another framework's memory budget, where a caching allocator already
// holds the device memory and a fresh cudaMalloc would fail or fragment it.
// Others sit on a latency-critical path where cudaMalloc's implicit device
// synchronisation is not acceptable.  This entry point allocates nothing; the
// scratch lives in `g_noalloc_scratch` below, which every GPU that loads the
// library keeps for the life of the process.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "q4_internal.h"

namespace {

constexpr int64_t kScratchBytes = Q4ADAMW_NOALLOC_SCRATCH_BYTES;

// File-scope device scratch.  In host code this name is only a host-side
// stand-in: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per
// device (with that device current).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return (int)e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return 0;
}

}  // namespace

extern "C" int q4adamw_step_noalloc(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                                    float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags,
                                    void* stream) {
    int64_t need = 0;
    if (int rc = q4adamw_workspace_bytes(t, n, recipe, &need)) return rc;
    if (need > kScratchBytes) return Q4_EWORKSPACE;
    void* ws = nullptr;
    if (int ce = scratch_address(&ws)) return q4::record_cuda_error(ce);
    return q4adamw_step(t, n, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, ws, kScratchBytes,
                        stream);
}

extern "C" int q4adamw_step_noalloc_status(uint32_t* status, void* stream) {
    if (!status) return Q4_EINVAL;
    void* ws = nullptr;
    if (int ce = scratch_address(&ws)) return q4::record_cuda_error(ce);
    return q4adamw_step_status(ws, status, stream);
}
