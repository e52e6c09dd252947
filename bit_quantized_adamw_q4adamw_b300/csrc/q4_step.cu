// Fused 4-bit AdamW step kernel for sm_103a.
//
// One warp processes one pair of consecutive 128-element blocks of a tensor:
// lanes 0-15 own block 2p, lanes 16-31 block 2p+1, and lane j of a half owns
// the 8 consecutive elements 8j..8j+7 of its block.  Per lane the step loads
// 16 B of BF16 gradient, 32 B of FP32 master weight and one 32-bit word of m
// codes and of v codes; per block one FP32 scale of m and of v.  It writes the
// same amounts back plus 16 B of BF16 weights.  Block reductions (absmax, the
// EDEN sums) are half-warp shuffles; per-block tables (dequantisation levels,
// scaled thresholds and levels, ZIP-SR preconditioner levels) are built by the
// 16 lanes of a half in shared memory and read by table lookup.
//
// The grid is persistent: warps stride over the global list of block pairs of
// all tensors (tensor-chunk table = prefix sums of pairs per tensor); a warp's
// pairs increase monotonically, so its tensor index only moves forward.
//
// The arithmetic follows the per-element and per-block definitions of the
// method (listing page "Rounding in Preconditioner Space", Abstract and
// Tables 1-2; news page paragraphs 2-4; AReno docs "State representation")
// operation by operation in FP32 with round-to-nearest intrinsics, so that
// codes and scales are bit-identical to a plain sequential evaluation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"

namespace q4 {
namespace {

constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: adding it rounds to an integer in the low mantissa bits
constexpr float kTwoM24 = 5.9604644775390625e-08f;   // 2^-24

struct __align__(16) WarpTables {
    float deqm[32];   // [half][16] NF4 level * old s_m
    float deqv[32];   // [half][16] v level * old s_v
    float tm[32];     // [half][16] NF4 threshold * new s_m
    float am[32];     // [half][16] NF4 level * new s_m (LM-head SR)
    float av[32];     // [half][16] v level * new s_v (ZIP-SR) or v threshold * new s_v (RTN)
    float2 rd[32];    // [half][16] (r_k, (r_k - r_{k+1}) * 2^-24) for ZIP-SR
};

struct SmemAll {
    float vl[16];     // unscaled v levels (EDEN reconstruction)
    uint8_t lut_nf4_t[64];
    uint8_t lut_nf4_l[64];
    uint8_t lut_v_l[kVLut];
    uint8_t lut_v_t[kVLut];
    WarpTables w[kWarps];
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t to_bf16(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Philox4x32-10 (Salmon et al., SC'11) with a precomputed key schedule.
__device__ __forceinline__ uint4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, const uint32_t* rk) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ rk[2 * r];
        const uint32_t n2 = hi0 ^ c3 ^ rk[2 * r + 1];
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return make_uint4(c0, c1, c2, c3);
}

// The 8 draws of elements idx..idx+7 (idx a multiple of 4) for `purpose`.
__device__ __forceinline__ void draws8(uint64_t idx, uint32_t purpose, uint32_t tensor_id, uint32_t step,
                                       const uint32_t* rk, uint32_t w[8]) {
    const uint64_t i1 = idx + 4;
    const uint4 a = philox((uint32_t)(idx >> 2), (uint32_t)(idx >> 34) | (purpose << 28), tensor_id, step, rk);
    const uint4 b = philox((uint32_t)(i1 >> 2), (uint32_t)(i1 >> 34) | (purpose << 28), tensor_id, step, rk);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

__device__ __forceinline__ float half_max(float x) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Fast candidate paths need a scale whose reciprocal and scaled tables are
// normal numbers; anything else (0, subnormal, huge, NaN) takes the exact
// sequential search.
__device__ __forceinline__ bool scale_in_fast_range(float s) { return s >= 0x1p-90f && s <= 0x1p90f; }

// Per-element core shared by every recipe.  Returns r = 1/(sqrt(v')*c2+eps).
__device__ __forceinline__ void adamw_core(const StepParams& P, float g, float m, float v, float& theta, float& m1,
                                           float& v1, float& r, bool fact, float vhat) {
    m1 = __fmaf_rn(P.beta1, m, __fmul_rn(P.omb1, g));
    v1 = fact ? vhat : __fmaf_rn(P.beta2, v, __fmul_rn(P.omb2, __fmul_rn(g, g)));
    r = __frcp_rn(__fadd_rn(__fmul_rn(__fsqrt_rn(v1), P.c2), P.eps));
    theta = __fsub_rn(__fmul_rn(theta, P.decay), __fmul_rn(P.step_size, __fmul_rn(m1, r)));
}

template <int RECIPE>
__device__ __forceinline__ void process_pair(const StepParams& P, const DevTensor& d, int64_t pair, int lane,
                                             SmemAll& sm, const float my_nf4, const float my_nf4t,
                                             const float my_vl, const float my_vt) {
    WarpTables& wt = sm.w[threadIdx.x >> 5];
    const int half = lane >> 4, j = lane & 15, hb = half * 16;
    const int64_t nblk = (d.numel + kBlock - 1) / kBlock;
    const int64_t blk = pair * 2 + half;
    const bool blk_ok = blk < nblk;
    const int64_t e0 = blk * kBlock + j * 8;
    const int64_t rem = d.numel - e0;
    const int nvalid = rem >= 8 ? 8 : (rem > 0 ? (int)rem : 0);
    const bool fact = (RECIPE == Q4_RECIPE_FACTORED) && (d.flags & DF_FACTORED);
    const bool m_sr = (d.flags & DF_M_SR) != 0;

    // ---- loads -------------------------------------------------------
    float g[8], th[8];
    uint32_t qmw = 0, qvw = 0;
    float sm_old = 0.f, sv_old = 0.f;
    if (blk_ok) {
        sm_old = __ldg(d.ms + blk);
        qmw = __ldg(reinterpret_cast<const uint32_t*>(d.mc + blk * 64) + j);
        if (!fact) {
            sv_old = __ldg(d.vs + blk);
            qvw = __ldg(reinterpret_cast<const uint32_t*>(d.vc + blk * 64) + j);
        }
    }
    if (nvalid == 8) {
        const uint4 gw = __ldcs(reinterpret_cast<const uint4*>(d.grad + e0));
        const float4 t0 = __ldcs(reinterpret_cast<const float4*>(d.param + e0));
        const float4 t1 = __ldcs(reinterpret_cast<const float4*>(d.param + e0 + 4));
        g[0] = bf16lo(gw.x); g[1] = bf16hi(gw.x); g[2] = bf16lo(gw.y); g[3] = bf16hi(gw.y);
        g[4] = bf16lo(gw.z); g[5] = bf16hi(gw.z); g[6] = bf16lo(gw.w); g[7] = bf16hi(gw.w);
        th[0] = t0.x; th[1] = t0.y; th[2] = t0.z; th[3] = t0.w;
        th[4] = t1.x; th[5] = t1.y; th[6] = t1.z; th[7] = t1.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            g[i] = 0.f;
            th[i] = 0.f;
            if (i < nvalid) {
                g[i] = __uint_as_float((uint32_t)d.grad[e0 + i] << 16);
                th[i] = d.param[e0 + i];
            }
        }
    }

    // ---- dequantisation tables (old scales) ---------------------------
    wt.deqm[hb + j] = __fmul_rn(my_nf4, sm_old);
    if (!fact) wt.deqv[hb + j] = __fmul_rn(my_vl, sv_old);
    __syncwarp();

    // factored second moment: vhat = R_i * C_j / mean(R)
    float rbar = 0.f;
    int64_t frow = 0, fcol = 0;
    if (fact) {
        rbar = __ldg(d.rbar);
        if (nvalid > 0) {
            frow = e0 / d.cols;
            fcol = e0 - frow * d.cols;
        }
    }

    // ---- per-element AdamW --------------------------------------------
    float m1[8], v1[8], r[8];
    float amax = 0.f, vmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float m = wt.deqm[hb + ((qmw >> (4 * i)) & 15u)];
        float v = 0.f, vhat = 0.f;
        if (fact) {
            if (i < nvalid) {
                const float R = __ldg(d.vrow + frow), C = __ldg(d.vcol + fcol);
                vhat = (rbar == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(R, C), rbar);
                if (++fcol == d.cols) { fcol = 0; ++frow; }
            }
        } else {
            v = wt.deqv[hb + ((qvw >> (4 * i)) & 15u)];
        }
        adamw_core(P, g[i], m, v, th[i], m1[i], v1[i], r[i], fact, vhat);
        if (i >= nvalid) { m1[i] = 0.f; v1[i] = 0.f; }
        amax = fmaxf(amax, fabsf(m1[i]));
        vmax = fmaxf(vmax, fabsf(v1[i]));
    }

    // ---- weights out ----------------------------------------------------
    if (nvalid == 8) {
        __stcs(reinterpret_cast<float4*>(d.param + e0), make_float4(th[0], th[1], th[2], th[3]));
        __stcs(reinterpret_cast<float4*>(d.param + e0 + 4), make_float4(th[4], th[5], th[6], th[7]));
        if (d.flags & DF_BF16) {
            uint4 o;
            o.x = pack_bf16x2(th[0], th[1]);
            o.y = pack_bf16x2(th[2], th[3]);
            o.z = pack_bf16x2(th[4], th[5]);
            o.w = pack_bf16x2(th[6], th[7]);
            __stcs(reinterpret_cast<uint4*>(d.bf16 + e0), o);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < nvalid) {
                d.param[e0 + i] = th[i];
                if (d.flags & DF_BF16) d.bf16[e0 + i] = to_bf16(th[i]);
            }
        }
    }

    // ---- block scales -----------------------------------------------------
    const float s_m = half_max(amax);
    const float s_v = fact ? 0.f : half_max(vmax);

    // ---- requantisation tables (new scales) ----------------------------
    wt.tm[hb + j] = __fmul_rn(my_nf4t, s_m);
    if (m_sr) wt.am[hb + j] = __fmul_rn(my_nf4, s_m);
    if (RECIPE == Q4_RECIPE_ZIP_SR) {
        const float a = __fmul_rn(my_vl, s_v);
        const float rk = __frcp_rn(__fadd_rn(__fmul_rn(__fsqrt_rn(a), P.c2), P.eps));
        const float rk1 = __shfl_down_sync(0xffffffffu, rk, 1);
        wt.av[hb + j] = a;
        wt.rd[hb + j] = make_float2(rk, j < 15 ? __fmul_rn(__fsub_rn(rk, rk1), kTwoM24) : 0.f);
    } else if (!fact) {
        wt.av[hb + j] = __fmul_rn(my_vt, s_v);
    }
    __syncwarp();

    // ---- m codes ----------------------------------------------------------
    uint32_t cm = 0;
    {
        const bool fast = scale_in_fast_range(s_m);
        const float rho16 = __fmul_rn(16.f, __frcp_rn(s_m));
        uint32_t w[8];
        if (m_sr) draws8(d.elem_offset + (uint64_t)e0, 0u, d.tensor_id, P.step, P.round_keys, w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float x = m1[i];
            int code;
            if (!m_sr) {
                if (fast) {
                    const uint32_t bi = __float_as_uint(__fmaf_rn(x, rho16, kMagic + 16.f)) & 63u;
                    const int c = sm.lut_nf4_t[bi];
                    code = c + (x > wt.tm[hb + c] ? 1 : 0);
                } else {
                    code = 0;
#pragma unroll 1
                    for (int k = 0; k < 15; ++k) code += (x > wt.tm[hb + k]) ? 1 : 0;
                }
            } else {
                int k;
                if (fast) {
                    const uint32_t bi = __float_as_uint(__fmaf_rn(x, rho16, kMagic + 16.f)) & 63u;
                    const int c = sm.lut_nf4_l[bi];
                    k = c + (wt.am[hb + c + 1] <= x ? 1 : 0);
                } else {
                    k = 0;
#pragma unroll 1
                    for (int q = 0; q < 16; ++q)
                        if (wt.am[hb + q] <= x) k = q;
                }
                if (k < 15) {
                    const float ak = wt.am[hb + k], ak1 = wt.am[hb + k + 1];
                    const float u = __fmul_rn((float)(w[i] >> 8), kTwoM24);
                    code = k + (__fmul_rn(u, __fsub_rn(ak1, ak)) < __fsub_rn(x, ak) ? 1 : 0);
                } else {
                    code = 15;
                }
            }
            if (i >= nvalid) code = 0;
            cm |= (uint32_t)code << (4 * i);
        }
    }

    // ---- v codes ----------------------------------------------------------
    uint32_t cv = 0;
    float sv_store = s_v;
    if (!fact) {
        const bool fast = scale_in_fast_range(s_v);
        const float rho = __frcp_rn(s_v);
        if (RECIPE == Q4_RECIPE_ZIP_SR) {
            uint32_t w[8];
            draws8(d.elem_offset + (uint64_t)e0, 1u, d.tensor_id, P.step, P.round_keys, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = v1[i];
                int k;
                if (fast) {
                    const uint32_t bi = min(__float_as_uint(__fmul_rn(fabsf(x), rho)) >> 19, (uint32_t)(kVLut - 1));
                    const int c = sm.lut_v_l[bi];
                    k = c + (wt.av[hb + c + 1] <= x ? 1 : 0);
                } else {
                    k = 0;
#pragma unroll 1
                    for (int q = 0; q < 16; ++q)
                        if (wt.av[hb + q] <= x) k = q;
                }
                const float2 e = wt.rd[hb + k];
                // u * (r_k - r_{k+1}) with u = (w >> 8) 2^-24, as (w >> 8) * ((r_k - r_{k+1}) 2^-24)
                int code = k + (__fmul_rn((float)(w[i] >> 8), e.y) < __fsub_rn(e.x, r[i]) ? 1 : 0);
                if (i >= nvalid) code = 0;
                cv |= (uint32_t)code << (4 * i);
            }
        } else {
            int q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = v1[i];
                int code;
                if (fast) {
                    const uint32_t bi = min(__float_as_uint(__fmul_rn(fabsf(x), rho)) >> 19, (uint32_t)(kVLut - 1));
                    const int c = sm.lut_v_t[bi];
                    code = c + (x > wt.av[hb + c] ? 1 : 0);
                } else {
                    code = 0;
#pragma unroll 1
                    for (int k = 0; k < 15; ++k) code += (x > wt.av[hb + k]) ? 1 : 0;
                }
                if (i >= nvalid) code = 0;
                q[i] = code;
                cv |= (uint32_t)code << (4 * i);
            }
            if (RECIPE == Q4_RECIPE_ZE_EDEN) {
                // EDEN scale s * |y|^2 / <y, L[q]>, y = v' * (1/s), fixed summation
                // order.  The sums run on every lane (the shuffles need the whole
                // warp); blocks with s below the smallest normal keep s.
                float pa[2], pb[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float sa = 0.f, sb = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e = 4 * h + i;
                        const float y = __fmul_rn(v1[e], rho);
                        const float yh = sm.vl[q[e]];
                        const float ta = __fmul_rn(y, y), tb = __fmul_rn(y, yh);
                        sa = (i == 0) ? ta : __fadd_rn(sa, ta);
                        sb = (i == 0) ? tb : __fadd_rn(sb, tb);
                    }
                    pa[h] = sa;
                    pb[h] = sb;
                }
                float A = __fadd_rn(pa[0], pa[1]);
                float B = __fadd_rn(pb[0], pb[1]);
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    A = __fadd_rn(A, __shfl_xor_sync(0xffffffffu, A, o));
                    B = __fadd_rn(B, __shfl_xor_sync(0xffffffffu, B, o));
                }
                if (s_v >= 0x1p-126f) sv_store = (B == 0.f) ? 0.f : __fmul_rn(s_v, __fdiv_rn(A, B));
            }
        }
    }

    // ---- codes and scales out --------------------------------------------
    if (blk_ok) {
        reinterpret_cast<uint32_t*>(d.mc + blk * 64)[j] = cm;
        if (!fact) reinterpret_cast<uint32_t*>(d.vc + blk * 64)[j] = cv;
        if (j == 0) {
            d.ms[blk] = s_m;
            if (!fact) d.vs[blk] = sv_store;
        }
    }
    __syncwarp();
}

template <int RECIPE>
__global__ void __launch_bounds__(kThreads) step_kernel(const __grid_constant__ StepParams P) {
    __shared__ SmemAll sm;
    if (threadIdx.x < 16) sm.vl[threadIdx.x] = P.tab.vl[threadIdx.x];
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        sm.lut_nf4_t[i] = P.tab.lut_nf4_t[i];
        sm.lut_nf4_l[i] = P.tab.lut_nf4_l[i];
    }
    for (int i = threadIdx.x; i < kVLut / 4; i += blockDim.x) {
        reinterpret_cast<uint32_t*>(sm.lut_v_l)[i] = reinterpret_cast<const uint32_t*>(P.tab.lut_v_l)[i];
        reinterpret_cast<uint32_t*>(sm.lut_v_t)[i] = reinterpret_cast<const uint32_t*>(P.tab.lut_v_t)[i];
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int j = lane & 15;
    const float my_nf4 = P.tab.nf4[j], my_nf4t = P.tab.nf4_t[j];
    const float my_vl = P.tab.vl[j], my_vt = P.tab.vt[j];

    const int64_t W = (int64_t)gridDim.x * kWarps;
    int t = 0;
    int loaded = -1;
    DevTensor d;
    for (int64_t pair = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); pair < P.total_pairs; pair += W) {
        while (pair >= __ldg(P.pair_prefix + t + 1)) ++t;
        if (t != loaded) {
            d = P.tensors[t];
            loaded = t;
        }
        process_pair<RECIPE>(P, d, pair - __ldg(P.pair_prefix + t), lane, sm, my_nf4, my_nf4t, my_vl, my_vt);
    }
}

}  // namespace

int step_grid_size(int device, int64_t total_pairs) {
    static int cached_sms[64] = {0};
    static int cached_occ[64] = {0};
    if (device < 0 || device >= 64) device = 0;
    if (cached_sms[device] == 0) {
        int sms = 0, occ = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, step_kernel<Q4_RECIPE_ZIP_SR>, kThreads, 0);
        cached_sms[device] = sms > 0 ? sms : 1;
        cached_occ[device] = occ > 0 ? occ : 1;
    }
    const int64_t full = (int64_t)cached_sms[device] * cached_occ[device];
    const int64_t need = (total_pairs + kWarps - 1) / kWarps;
    return (int)(need < full ? (need > 0 ? need : 1) : full);
}

int launch_step(const StepParams& p, int grid, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (p.recipe) {
        case Q4_RECIPE_ZIP_SR: step_kernel<Q4_RECIPE_ZIP_SR><<<grid, kThreads, 0, s>>>(p); break;
        case Q4_RECIPE_ZE_EDEN: step_kernel<Q4_RECIPE_ZE_EDEN><<<grid, kThreads, 0, s>>>(p); break;
        default: step_kernel<Q4_RECIPE_FACTORED><<<grid, kThreads, 0, s>>>(p); break;
    }
    return (int)cudaGetLastError();
}

}  // namespace q4
