// Deterministic reductions shared by the factored-statistics and the decoding
// kernels of the q4adamw library.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace q4 {

// Mean of R[0..rows) by one CTA of exactly 256 threads in a fixed order:
// thread t sums R[t], R[t+256], ... left to right, then a binary tree over the
// 256 partials; the sum is divided by rows.  Every CTA that calls it on the
// same R gets the same bits.  All 256 threads must call it.
__device__ __forceinline__ float block_mean(const float* R, int64_t rows, float* red) {
    float acc = 0.f;
    for (int64_t i = threadIdx.x; i < rows; i += 256) acc = __fadd_rn(acc, R[i]);
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] = __fadd_rn(red[threadIdx.x], red[threadIdx.x + o]);
        __syncthreads();
    }
    const float mean = __fdiv_rn(red[0], (float)rows);
    __syncthreads();
    return mean;
}

}  // namespace q4
