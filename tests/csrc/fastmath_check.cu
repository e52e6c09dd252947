// Exhaustive GPU check of the step kernel's correctly rounded square root and
// reciprocal (scalar and paired forms) against CUDA's IEEE intrinsics
// (__fsqrt_rn, __frcp_rn), and a
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

// Paired versions: component 0 takes input i, component 1 input i ^ 1 (every
// input appears in both lanes of some pair).
__global__ void sqrt2_kernel(uint64_t lo, uint64_t hi, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += stride) {
        const float x0 = __uint_as_float((unsigned)i), x1 = __uint_as_float((unsigned)i ^ 1u);
        if (!q4::sqrt_fast_domain(x0) || !q4::sqrt_fast_domain(x1)) continue;
        const float2 s = q4::sqrt2_rn_normal(make_float2(x0, x1));
        if (!same(s.x, __fsqrt_rn(x0)) || !same(s.y, __fsqrt_rn(x1))) record(count, first, (unsigned)i);
    }
}

__global__ void rcp2_kernel(uint64_t lo, uint64_t hi, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += stride) {
        const float d0 = __uint_as_float((unsigned)i), d1 = __uint_as_float((unsigned)i ^ 1u);
        const float2 y = q4::rcp2_rn_normal(make_float2(d0, d1));
        if (!same(y.x, __frcp_rn(d0)) || !same(y.y, __frcp_rn(d1))) record(count, first, (unsigned)i);
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

// The paired quotient (two dividends, one divisor) against __fdiv_rn, on the
// same operand distribution as div_kernel; the second dividend is the first
// scaled by a random power of two in [2^-8, 2^8] (both kept in range).
__global__ void div2_kernel(uint64_t n, uint64_t seed, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t u0 = mix(seed * 0x100000000ull + 2 * i), u1 = mix(seed * 0x100000000ull + 2 * i + 1);
        const uint32_t ea = 35 + (u0 >> 24) % 185, eb = 27 + (u1 >> 24) % 201;
        uint32_t mb = u1 & 0x7fffffu;
        if ((i & 3) == 1) mb = 0x7fffffu;
        const float b = __uint_as_float((eb << 23) | mb);
        float a = __uint_as_float((ea << 23) | (u0 & 0x7fffffu));
        if ((i & 3) == 2) a = __uint_as_float(__float_as_uint(__fmul_rn(b, (float)(1 + (u0 & 255)))) + (u0 >> 8 & 3) - 1);
        const float a2 = __uint_as_float(__float_as_uint(a) + ((int)((u1 >> 8) % 17) - 8) * (1 << 23));
        const float q1 = __fdiv_rn(a, b), q2 = __fdiv_rn(a2, b);
        const bool in1 = fabsf(q1) >= 0x1p-100f && fabsf(q1) <= 0x1p100f && fabsf(a) >= 0x1p-100f && fabsf(a) <= 0x1p100f;
        const bool in2 = fabsf(q2) >= 0x1p-100f && fabsf(q2) <= 0x1p100f && fabsf(a2) >= 0x1p-100f && fabsf(a2) <= 0x1p100f;
        if (!in1 || !in2) continue;
        const float2 q = q4::div2_rn_by_rcp(make_float2(a, a2), b, __frcp_rn(b));
        if (!same(q.x, q1) || !same(q.y, q2)) record(count, first, (unsigned)(i & 0xffffffffu));
    }
}

// The paired-arithmetic patterns the step kernel relies on, each against the
// scalar operations: paired mul, add and fma alone; a single-use paired product
// finished by a scalar add; a single-use paired product as the addend of a
// paired fma.  (A single-use paired product feeding a paired add may be fused
// by the compiler; the kernel never uses that pattern.)
__global__ void pair_ops_kernel(uint64_t n, uint64_t seed, unsigned long long* count, unsigned* first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t u0 = mix(seed * 0x100000000ull + 3 * i), u1 = mix(seed * 0x100000000ull + 3 * i + 1);
        const uint32_t u2 = mix(seed * 0x100000000ull + 3 * i + 2);
        const float a = __uint_as_float(((90u + (u0 >> 26)) << 23) | (u0 & 0x7fffffu));
        const float b = __uint_as_float(((90u + (u1 >> 26)) << 23) | (u1 & 0x7fffffu));
        const float c = __uint_as_float(((110u + (u2 >> 27)) << 23) | (u2 & 0x7fffffu) | ((u2 & 0x4000000u) << 5));
        const float2 m = q4::mul2_rn(make_float2(a, b), make_float2(b, c));
        const float2 s = q4::add2_rn(make_float2(a, b), make_float2(c, -c));
        const float2 f = q4::fma2_rn(make_float2(a, b), make_float2(c, a), make_float2(b, c));
        const float2 pm = q4::mul2_rn(make_float2(a, b), make_float2(b, a));
        const float2 p = make_float2(__fadd_rn(pm.x, c), __fadd_rn(pm.y, -c));
        const float2 fm = q4::fma2_rn(make_float2(c, b), make_float2(b, c), q4::mul2_rn(make_float2(a, c), make_float2(c, a)));
        const bool bad = !same(m.x, __fmul_rn(a, b)) || !same(m.y, __fmul_rn(b, c)) ||
                         !same(s.x, __fadd_rn(a, c)) || !same(s.y, __fadd_rn(b, -c)) ||
                         !same(f.x, __fmaf_rn(a, c, b)) || !same(f.y, __fmaf_rn(b, a, c)) ||
                         !same(p.x, __fadd_rn(__fmul_rn(a, b), c)) || !same(p.y, __fadd_rn(__fmul_rn(b, a), -c)) ||
                         !same(fm.x, __fmaf_rn(c, b, __fmul_rn(a, c))) || !same(fm.y, __fmaf_rn(b, c, __fmul_rn(c, a)));
        if (bad) record(count, first, (unsigned)(i & 0xffffffffu));
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
        case 21: div2_kernel<<<grid, block, 0, s>>>(hi, lo, count, first); break;
        case 30: sqrt2_kernel<<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 31: rcp2_kernel<<<grid, block, 0, s>>>(lo, hi, count, first); break;
        case 40: pair_ops_kernel<<<grid, block, 0, s>>>(hi, lo, count, first); break;
        default: return -1;
    }
    return (int)cudaGetLastError();
}
