// Exhaustive GPU check of the step kernel's correctly rounded square root and
// reciprocal against CUDA's IEEE intrinsics (__fsqrt_rn, __frcp_rn), and a
// randomised check of the reciprocal-based quotient against __fdiv_rn.
// Test infrastructure: built and loaded by tests/test_gpu_fastmath.py.
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_fastmath.cuh"

namespace {

__device__ __forceinline__ bool same(float a, float b) {
    return __float_as_uint(a) == __float_as_uint(b) || (a != a && b != b);
}

__device__ __forceinline__ void record(unsigned long long* count, unsigned* first, unsigned bits) {
    atomicAdd(count, 1ull);
    atomicMin(first, bits);
}

template <int V>
__global__ void sqrt_kernel(uint64_t lo, uint64_t hi, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += stride) {
        const float x = __uint_as_float((unsigned)i);
        if (!q4::sqrt_fast_domain(x)) continue;
        if (!same(q4::sqrt_rn_normal<V>(x), __fsqrt_rn(x))) record(count, first, (unsigned)i);
    }
}

template <int V>
__global__ void rcp_kernel(uint64_t lo, uint64_t hi, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += stride) {
        const float d = __uint_as_float((unsigned)i);
        if (!same(q4::rcp_rn_normal<V>(d), __frcp_rn(d))) record(count, first, (unsigned)i);
    }
}

__device__ __forceinline__ uint32_t mix(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)(z ^ (z >> 31));
}

// Random (a, b) with exponents in [-100, 100]; every fourth b has an all-ones
// significand and every fourth a sits next to a multiple of b.
__global__ void div_kernel(uint64_t n, uint64_t seed, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t u0 = mix(seed * 0x100000000ull + 2 * i), u1 = mix(seed * 0x100000000ull + 2 * i + 1);
        const uint32_t ea = 27 + (u0 >> 24) % 201, eb = 27 + (u1 >> 24) % 201;
        uint32_t mb = u1 & 0x7fffffu;
        if ((i & 3) == 1) mb = 0x7fffffu;
        const float b = __uint_as_float((eb << 23) | mb);
        float a = __uint_as_float((ea << 23) | (u0 & 0x7fffffu));
        if ((i & 3) == 2) a = __uint_as_float(__float_as_uint(__fmul_rn(b, (float)(1 + (u0 & 255)))) + (u0 >> 8 & 3) - 1);
        if (u0 & 0x800000u) a = -a;
        const float q = __fdiv_rn(a, b);
        const float aq = fabsf(q);
        if (!(aq >= 0x1p-100f && aq <= 0x1p100f) || !(fabsf(a) >= 0x1p-100f && fabsf(a) <= 0x1p100f)) continue;
        if (!same(q4::div_rn_by_rcp(a, b, __frcp_rn(b)), q)) record(count, first, (unsigned)(i & 0xffffffffu));
    }
}

}  // namespace

extern "C" int fm_check(int which, int variant, uint64_t lo, uint64_t hi, unsigned long long* count,
                        unsigned* first, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = 148 * 8, block = 256;
    switch (which * 10 + variant) {
        case 0: sqrt_kernel<0><<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 1: sqrt_kernel<1><<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 11: rcp_kernel<1><<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 12: rcp_kernel<2><<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 20: div_kernel<<<grid, block, 0, s>>>(hi, lo, count, first); break;
        default: return -1;
    }
    return (int)cudaGetLastError();
}
