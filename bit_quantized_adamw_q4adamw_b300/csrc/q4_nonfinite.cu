// Count of non-finite BF16 gradients (NaN, +inf, -inf) over a tensor list:
// an optional check a caller runs before a step, for instance to skip a step
// whose gradients overflowed.  One pass over the gradients (2 bytes per
// element): a grid-stride loop over the concatenated element list in runs of
// 8 elements (one 16-byte load where the run is whole and aligned), a warp
// sum, and one atomic add per warp into the caller's 64-bit device word,
// which the call zeroes first.  A BF16 value is non-finite when its exponent
// bits are all ones.
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_reduce.cuh"

namespace q4 {
namespace {

constexpr int kNfThreads = 256;

__device__ __forceinline__ uint32_t nonfinite_pair(uint32_t w) {
    // two BF16 values in one word: exponent field all ones in either half
    return ((w & 0x7f80u) == 0x7f80u ? 1u : 0u) + ((w & 0x7f800000u) == 0x7f800000u ? 1u : 0u);
}

__global__ void __launch_bounds__(kNfThreads) nonfinite_kernel(const __grid_constant__ NonfiniteParams P) {
    unsigned long long cnt = 0;
    const int64_t stride = (int64_t)gridDim.x * kNfThreads;
    for (int64_t r = (int64_t)blockIdx.x * kNfThreads + threadIdx.x; r < P.total_runs; r += stride) {
        const int t = find_tensor(P.run_prefix, P.n_tensors, r);
        const NormTensor& d = P.tensors[t];
        const int64_t e0 = (r - __ldg(P.run_prefix + t)) * 8;
        const int64_t left = d.numel - e0;
        if (left >= 8) {
            // grad is 16-byte aligned and e0 a multiple of 8: one vector load
            const uint4 w = __ldcs(reinterpret_cast<const uint4*>(d.grad + e0));
            cnt += nonfinite_pair(w.x) + nonfinite_pair(w.y) + nonfinite_pair(w.z) + nonfinite_pair(w.w);
        } else {
            for (int64_t k = 0; k < left; ++k) cnt += (d.grad[e0 + k] & 0x7f80u) == 0x7f80u ? 1u : 0u;
        }
    }
    // a thread counts at most 8 per run it visits, so the warp's 32-bit sum is
    // exact below 2^24 runs per thread (about 4e13 elements at the launch's
    // ~3e5 threads), far beyond any device memory
    const uint32_t warp_cnt = __reduce_add_sync(0xffffffffu, (uint32_t)cnt);
    if ((threadIdx.x & 31) == 0 && warp_cnt) atomicAdd(P.out, (unsigned long long)warp_cnt);
}

}  // namespace

int launch_nonfinite(const NonfiniteParams& p, int device, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(p.out, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return (int)e;
    if (p.total_runs == 0) return 0;
    int sms = 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) sms = 148;
    int64_t grid = (p.total_runs + kNfThreads - 1) / kNfThreads;
    if (grid > (int64_t)sms * 8) grid = (int64_t)sms * 8;
    nonfinite_kernel<<<(int)grid, kNfThreads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
