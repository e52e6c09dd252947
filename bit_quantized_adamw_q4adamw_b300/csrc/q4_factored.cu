// Factored second-moment statistics for rank >= 2 tensors (AReno docs
// "4-bit AdamW", section "State representation": Adafactor-style row and
// column means of g^2 over the [shape[0], -1] view, kept as exponential
// averages; 1-D tensors keep packed 4-bit v).
//
// Three passes, all multi-tensor and deterministic (fixed summation order, no
// atomics):
//   row_kernel     one warp per row: FP32 sum of g^2 along the row (each lane a
//                  strided partial, then a warp tree), R_i <- beta2 R_i +
//                  (1-beta2) * sum/cols.
//   colpart_kernel one CTA per (tensor, 64-row slab, 2048-column segment): each
//                  thread sums g^2 of 8 columns down the slab and writes the
//                  slab's partial column sums.
//   colfin_kernel  one thread per column: sums the slab partials in slab order,
//                  C_j <- beta2 C_j + (1-beta2) * sum/rows.
//   rbar_kernel    one CTA per factored tensor: mean(R) in a fixed tree order,
//                  stored with its correctly rounded reciprocal.
// The step kernel then reads vhat_ij = R_i * C_j / mean(R).
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_reduce.cuh"

namespace q4 {

// Index of the tensor whose prefix range [prefix[t], prefix[t+1]) holds idx.
__device__ __forceinline__ int find_tensor(const int64_t* prefix, int n, int64_t idx) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(prefix + mid) <= idx) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float sq_bf16(uint16_t h) {
    const float g = __uint_as_float((uint32_t)h << 16);
    return __fmul_rn(g, g);
}

namespace {

__global__ void __launch_bounds__(256) row_kernel(const __grid_constant__ FactoredParams P) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t W = (int64_t)gridDim.x * 8;
    for (int64_t row = gw; row < P.total_rows; row += W) {
        const int t = find_tensor(P.row_prefix, P.n_tensors, row);
        const DevTensor& d = P.tensors[t];
        const int64_t i = row - __ldg(P.row_prefix + t);
        const uint16_t* g = d.grad + i * d.cols;
        float acc = 0.f;
        for (int64_t c = lane; c < d.cols; c += 32) acc = __fadd_rn(acc, sq_bf16(g[c]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
        if (lane == 0) {
            const float mean = __fdiv_rn(acc, (float)d.cols);
            d.vrow[i] = __fmaf_rn(P.beta2, d.vrow[i], __fmul_rn(P.omb2, mean));
        }
    }
}

__global__ void __launch_bounds__(256) colpart_kernel(const __grid_constant__ FactoredParams P) {
    for (int64_t tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
        const int t = find_tensor(P.tile_prefix, P.n_tensors, tile);
        const DevTensor& d = P.tensors[t];
        const int64_t local = tile - __ldg(P.tile_prefix + t);
        const int64_t nseg = (d.cols + kSegCols - 1) / kSegCols;
        const int64_t slab = local / nseg, seg = local - slab * nseg;
        const int64_t c0 = seg * kSegCols + (int64_t)threadIdx.x * 8;
        const int64_t r0 = slab * kSlabRows;
        const int64_t r1 = (r0 + kSlabRows < d.rows) ? r0 + kSlabRows : d.rows;
        if (c0 >= d.cols) continue;
        const int nc = (d.cols - c0 >= 8) ? 8 : (int)(d.cols - c0);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int64_t r = r0; r < r1; ++r) {
            const uint16_t* g = d.grad + r * d.cols + c0;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < nc) acc[k] = __fadd_rn(acc[k], sq_bf16(g[k]));
        }
        float* out = d.colpart + slab * d.cols + c0;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < nc) out[k] = acc[k];
    }
}

__global__ void __launch_bounds__(256) colfin_kernel(const __grid_constant__ FactoredParams P) {
    for (int64_t col = (int64_t)blockIdx.x * 256 + threadIdx.x; col < P.total_cols;
         col += (int64_t)gridDim.x * 256) {
        const int t = find_tensor(P.col_prefix, P.n_tensors, col);
        const DevTensor& d = P.tensors[t];
        const int64_t j = col - __ldg(P.col_prefix + t);
        const int64_t nslab = (d.rows + kSlabRows - 1) / kSlabRows;
        float acc = 0.f;
        for (int64_t s = 0; s < nslab; ++s) acc = __fadd_rn(acc, __ldg(d.colpart + s * d.cols + j));
        const float mean = __fdiv_rn(acc, (float)d.rows);
        d.vcol[j] = __fmaf_rn(P.beta2, d.vcol[j], __fmul_rn(P.omb2, mean));
    }
}

__global__ void __launch_bounds__(256) rbar_kernel(const __grid_constant__ FactoredParams P) {
    __shared__ float red[256];
    for (int k = blockIdx.x; k < P.n_factored; k += gridDim.x) {
        const DevTensor& d = P.tensors[__ldg(P.factored_ids + k)];
        const float mean = block_mean(d.vrow, d.rows, red);
        if (threadIdx.x == 0) *reinterpret_cast<float2*>(d.rbar) = make_float2(mean, __frcp_rn(mean));
    }
}

int grid_for(int64_t work, int per_cta) {
    int64_t g = (work + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > 148 * 16) g = 148 * 16;
    return (int)g;
}

}  // namespace

int launch_factored(const FactoredParams& p, void* stream) {
    if (p.n_factored == 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    row_kernel<<<grid_for(p.total_rows, 8), 256, 0, s>>>(p);
    colpart_kernel<<<grid_for(p.total_tiles, 1), 256, 0, s>>>(p);
    colfin_kernel<<<grid_for(p.total_cols, 256), 256, 0, s>>>(p);
    rbar_kernel<<<p.n_factored < 1024 ? p.n_factored : 1024, 256, 0, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
