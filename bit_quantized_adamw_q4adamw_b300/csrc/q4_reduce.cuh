// Deterministic reductions and small helpers shared by the step, factored-
// statistics, gradient-norm and decoding kernels of the q4adamw library.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace q4 {

// Index of the tensor whose prefix range [prefix[t], prefix[t+1]) holds idx
// (the last such t when empty ranges share the start).
__device__ __forceinline__ int find_tensor(const int64_t* prefix, int n, int64_t idx) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(prefix + mid) <= idx) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Global-norm clipping factor from the device sum of squares (NULL: 1): the
// coefficient of torch.nn.utils.clip_grad_norm_, max_norm * (1 / (norm +
// 1e-6)) with each operation correctly rounded in FP32, clamped above at 1
// (a NaN sum gives NaN).
__device__ __forceinline__ float clip_factor(const float* sqnorm, float max_norm) {
    if (sqnorm == nullptr) return 1.f;
    const float norm = __fsqrt_rn(__ldg(sqnorm));
    const float c = __fmul_rn(max_norm, __frcp_rn(__fadd_rn(norm, 1e-6f)));
    return c >= 1.f ? 1.f : c;
}

// Mean of R[0..rows) by one CTA of exactly NT threads (a power of two) in a
// fixed order: thread t sums R[t], R[t+NT], ... left to right, then a binary
// tree over the NT partials; the sum is divided by rows.  Every CTA that
// calls it with the same NT on the same R gets the same bits.  All NT threads
// must call it; red holds NT floats.
template <int NT = 256>
__device__ __forceinline__ float block_mean(const float* R, int64_t rows, float* red) {
    float acc = 0.f;
    for (int64_t i = threadIdx.x; i < rows; i += NT) acc = __fadd_rn(acc, R[i]);
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int o = NT / 2; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] = __fadd_rn(red[threadIdx.x], red[threadIdx.x + o]);
        __syncthreads();
    }
    const float mean = __fdiv_rn(red[0], (float)rows);
    __syncthreads();
    return mean;
}

}  // namespace q4
