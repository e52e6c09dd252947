// Sum of squares of the BF16 gradients, the first half of global gradient-norm
// clipping (AReno docs "4-bit AdamW", section "State representation": gradient
// norm and clipping run directly on the BF16 gradient shards).  The clip
// factor itself is formed inside the step kernels (clip_factor in
// q4_reduce.cuh) and multiplies each FP32 gradient there.
//
// The result is bit-reproducible: per tensor it is recursive pairwise
// summation of the FP32 squares over the tensor padded with zeros to a power
// of two (adjacent pairs at every level), and the tensor sums are added left
// to right from 0.  Zero padding never changes a pairwise root (x + 0 = x for
// the non-negative squares), so any aligned power-of-two blocking yields the
// same bits; the kernels block it as
//   lane      8 consecutive elements (one 16-byte load), a 3-level tree;
//   tile      256 elements = 32 lanes, a 5-level lane tree;
//   group     32 tiles: each lane loads its 8 elements of 16 tiles at a time,
//             a transpose tree over offsets 1, 2, 4, 8 and one add at offset
//             16 leaves tile (lane & 15) of the half in every lane; the two
//             halves' tiles then meet in a 5-level butterfly;
//   chunk     8 groups per warp x 8 warps = 2048 tiles (512 Ki elements), one
//             CTA, written to partials[];
//   tensor    sqnorm_tensor_kernel: a tree over the chunk partials in aligned
//             blocks of 512, repeated until one value remains;
//   list      sqnorm_total_kernel: tensors left to right.
// Traffic: 2 bytes per element read once (ld.global.nc, no reuse), a few
// bytes per 512 Ki elements written.
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_reduce.cuh"

namespace q4 {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ld_nc_v4(const uint16_t* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float sq_lo(uint32_t w) {
    const float x = __uint_as_float(w << 16);
    return __fmul_rn(x, x);
}
__device__ __forceinline__ float sq_hi(uint32_t w) {
    const float x = __uint_as_float(w & 0xffff0000u);
    return __fmul_rn(x, x);
}

// Pairwise sum of the squares of 8 consecutive BF16 values.
__device__ __forceinline__ float lane_sum(const uint4 w) {
    return __fadd_rn(__fadd_rn(__fadd_rn(sq_lo(w.x), sq_hi(w.x)), __fadd_rn(sq_lo(w.y), sq_hi(w.y))),
                     __fadd_rn(__fadd_rn(sq_lo(w.z), sq_hi(w.z)), __fadd_rn(sq_lo(w.w), sq_hi(w.w))));
}

// Elements [e, e+8) of g with those at or past numel read as 0.
__device__ __forceinline__ uint4 load8(const uint16_t* g, int64_t numel, int64_t e) {
    if (e + 8 <= numel) return ld_nc_v4(g + e);
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = (e + k < numel) ? (uint32_t)__ldg(g + e + k) : 0u;
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

// Tile sums of tiles t0 .. t0+15 (t0 a multiple of 16): lane l returns the sum
// of tile t0 + (l & 15).
__device__ __forceinline__ float half_group(const uint16_t* g, int64_t numel, int64_t t0, int lane) {
    float q[16];
    const int64_t e0 = t0 * 256 + lane * 8;
    if ((t0 + 16) * 256 <= numel) {
        uint4 w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = ld_nc_v4(g + e0 + k * 256);
#pragma unroll
        for (int k = 0; k < 16; ++k) q[k] = lane_sum(w[k]);
    } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) q[k] = lane_sum(load8(g, numel, e0 + k * 256));
    }
    // transpose tree: after offset 2^s lane l holds, for the tiles whose low
    // s+1 index bits equal l's, the sum over the 2^(s+1) lanes sharing l's
    // higher bits
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const bool up = (lane >> s) & 1;
#pragma unroll
        for (int i = 0; i < (8 >> s); ++i) {
            const float keep = up ? q[2 * i + 1] : q[2 * i];
            const float send = up ? q[2 * i] : q[2 * i + 1];
            q[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 1 << s));
        }
    }
    return __fadd_rn(q[0], __shfl_xor_sync(kFull, q[0], 16));
}

// Sum of tiles t0 .. t0+31 of one tensor (t0 a multiple of 32), in every lane.
__device__ __forceinline__ float group_sum(const uint16_t* g, int64_t numel, int64_t t0, int lane) {
    const float a = half_group(g, numel, t0, lane);
    const float b = (t0 + 16) * 256 < numel ? half_group(g, numel, t0 + 16, lane) : 0.f;
    float x = lane < 16 ? a : b;        // lane l: tile t0 + l
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) x = __fadd_rn(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

__device__ __forceinline__ float tree8(const float* v) {
    return __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3])),
                     __fadd_rn(__fadd_rn(v[4], v[5]), __fadd_rn(v[6], v[7])));
}

__global__ void __launch_bounds__(kNormWarps * 32, 2) sqnorm_chunk_kernel(const __grid_constant__ NormParams P) {
    static_assert(kNormWarps == 8 && kNormGroupsPerWarp == 8, "tree8 reduces 8 groups and 8 warps");
    __shared__ float wsum[kNormWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t c = blockIdx.x; c < P.total_chunks; c += gridDim.x) {
        const int t = find_tensor(P.chunk_prefix, P.n_tensors, c);
        const NormTensor d = P.tensors[t];
        const int64_t tiles = (d.numel + 255) / 256;
        const int64_t wt0 = (c - __ldg(P.chunk_prefix + t)) * kNormChunkTiles + warp * (kNormGroupsPerWarp * 32);
        float gs[kNormGroupsPerWarp];
#pragma unroll
        for (int k = 0; k < kNormGroupsPerWarp; ++k) {
            const int64_t t0 = wt0 + k * 32;
            gs[k] = t0 < tiles ? group_sum(d.grad, d.numel, t0, lane) : 0.f;
        }
        const float w = tree8(gs);
        if (lane == 0) wsum[warp] = w;
        __syncthreads();
        if (threadIdx.x == 0) P.partials[c] = tree8(wsum);
        __syncthreads();
    }
}

constexpr int kTreeThreads = 256;   // reduces aligned blocks of 512 partials

__global__ void __launch_bounds__(kTreeThreads) sqnorm_tensor_kernel(const __grid_constant__ NormParams P) {
    __shared__ float red[kTreeThreads];
    const int tid = threadIdx.x;
    for (int t = blockIdx.x; t < P.n_tensors; t += gridDim.x) {
        float* a = P.partials + __ldg(P.chunk_prefix + t);
        int64_t k = __ldg(P.chunk_prefix + t + 1) - __ldg(P.chunk_prefix + t);
        // in place: block b's root goes to a[b], which lies in block 0 (read
        // before any root is written) or is a[0] itself
        while (k > 1) {
            const int64_t nb = (k + 2 * kTreeThreads - 1) / (2 * kTreeThreads);
            for (int64_t b = 0; b < nb; ++b) {
                const int64_t i = b * 2 * kTreeThreads + 2 * tid;
                const float x0 = i < k ? a[i] : 0.f;
                const float x1 = i + 1 < k ? a[i + 1] : 0.f;
                red[tid] = __fadd_rn(x0, x1);
                __syncthreads();
                for (int s = 1; s < kTreeThreads; s <<= 1) {
                    if ((tid & (2 * s - 1)) == 0) red[tid] = __fadd_rn(red[tid], red[tid + s]);
                    __syncthreads();
                }
                if (tid == 0) a[b] = red[0];
                __syncthreads();
            }
            k = nb;
        }
        if (tid == 0) P.tensor_sums[t] = k == 1 ? a[0] : 0.f;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kTreeThreads) sqnorm_total_kernel(const __grid_constant__ NormParams P) {
    __shared__ float buf[1024];
    float total = 0.f;
    for (int base = 0; base < P.n_tensors; base += 1024) {
        const int m = P.n_tensors - base < 1024 ? P.n_tensors - base : 1024;
        for (int i = threadIdx.x; i < m; i += kTreeThreads) buf[i] = P.tensor_sums[base + i];
        __syncthreads();
        if (threadIdx.x == 0)
            for (int i = 0; i < m; ++i) total = __fadd_rn(total, buf[i]);
        __syncthreads();
    }
    if (threadIdx.x == 0) *P.out = total;
}

}  // namespace

int launch_grad_sqnorm(const NormParams& p, int device, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int sms = 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) sms = 148;
    if (p.total_chunks > 0) {
        const int64_t cap = (int64_t)sms * 2;
        const int grid = (int)(p.total_chunks < cap ? p.total_chunks : cap);
        sqnorm_chunk_kernel<<<grid, kNormWarps * 32, 0, s>>>(p);
    }
    if (p.n_tensors > 0) {
        const int grid = p.n_tensors < 4096 ? p.n_tensors : 4096;
        sqnorm_tensor_kernel<<<grid, kTreeThreads, 0, s>>>(p);
    }
    sqnorm_total_kernel<<<1, kTreeThreads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
