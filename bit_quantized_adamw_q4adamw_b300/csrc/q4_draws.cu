// q4adamw_draws: the stochastic-rounding draws of the step, for checking and
// reproducing them.  The kernel evaluates the same device function the step
// kernel uses (q4_philox.cuh) for each requested element.
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_philox.cuh"

namespace q4 {
namespace {

struct DrawParams {
    uint32_t rk[20];
    uint64_t idx0;
    int64_t n;
    uint32_t step, tensor_id, purpose;
    uint32_t* out;
};

// One thread per group of four elements sharing a counter.
__global__ void __launch_bounds__(256) draws_kernel(const __grid_constant__ DrawParams P) {
    const uint64_t g0 = P.idx0 >> 2;
    const uint64_t g_last = (P.idx0 + (uint64_t)P.n - 1) >> 2;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t g = g0 + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g <= g_last; g += stride) {
        const uint64_t idx = g << 2;
        const uint4 w = philox((uint32_t)(idx >> 2), (uint32_t)(idx >> 34) | (P.purpose << 28), P.tensor_id, P.step,
                               P.rk);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint64_t e = idx + (uint64_t)k;
            if (e >= P.idx0 && e < P.idx0 + (uint64_t)P.n) P.out[e - P.idx0] = ww[k];
        }
    }
}

}  // namespace

int launch_draws(uint64_t seed, uint32_t step, uint32_t tensor_id, uint64_t idx0, uint32_t purpose, int64_t n,
                 uint32_t* out, void* stream) {
    DrawParams p{};
    philox_round_keys(seed, p.rk);
    p.idx0 = idx0;
    p.n = n;
    p.step = step;
    p.tensor_id = tensor_id;
    p.purpose = purpose;
    p.out = out;
    const int64_t groups = (int64_t)(((idx0 + (uint64_t)n - 1) >> 2) - (idx0 >> 2)) + 1;
    const int64_t blocks = (groups + 255) / 256;
    const int grid = (int)(blocks < 148 * 16 ? blocks : 148 * 16);
    draws_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
