// Fused 4-bit AdamW step kernel for sm_103a.
//
// Work unit: a tile = one pair of consecutive 128-element blocks of a tensor
// (256 parameters).  One warp computes one tile: lanes 0-15 own block 2p,
// lanes 16-31 block 2p+1, and lane j of a half owns the 8 consecutive
// elements 8j..8j+7 of its block.
//
// Data movement.  The grid is persistent (one 16-warp CTA per SM).  The global
// list of tiles of all tensors (the tensor-chunk table is the prefix sum of
// tiles per tensor) is cut into one contiguous range per warp; within a tensor
// each copy source advances by a constant per tile.  Each warp keeps two
// shared-memory stage buffers of three tiles each: while it computes the tiles
// of one, the next three are in flight.  A stage is filled by one pass of 24
// lanes, lanes 8g..8g+7 for its tile g, each group with its own cursor: per
// tile four cp.async.bulk copies (BF16 gradient, FP32 master weight, packed m
// and v code words; the tensor memory access unit moves whole 16-byte
// granules) and four 4-byte cp.async copies (the block scales, which are only
// 4-byte aligned), all completing on the stage's mbarrier, so a stage costs
// one wait and one issue pass for three tiles.  A tile whose length is
// not a multiple of 8 elements (a tensor's ragged tail) is read directly from
// global memory instead.  Results (FP32 and BF16 weights, codes, scales) are
// written straight from registers with coalesced streaming stores.  Every
// wait on an mbarrier is bounded by a clock limit (StepParams::wait_cycles,
// about one second by default); on expiry the warp sets ST_STAGE_TIMEOUT in
// the step's status word, drains its own copies, the late one included (each
// with the default limit), and exits.
//
// Arithmetic.  The method's per-element and per-block definitions (listing
// page "Rounding in Preconditioner Space", Abstract and Tables 1-2; news page
// paragraphs 2-4; AReno docs "State representation") are evaluated operation
// by operation in FP32 with round-to-nearest, so that codes, scales and
// weights are bit-identical to a plain sequential evaluation.  The square
// root and reciprocal of r = 1/(sqrt(v') c2 + eps) and the factored quotient
// use the correctly rounded sequences of q4_fastmath.cuh where a lane's
// inputs are inside their verified domains, and the IEEE intrinsics
// otherwise.  Block absmax is an integer warp reduction (redux.sync) on the
// bit patterns, the EDEN sums a fixed shuffle tree; per-block tables
// (dequantisation levels at the old scale, thresholds, levels and ZIP-SR
// preconditioner levels at the new scale) are built by the 16 lanes of a half
// in shared memory and read by table lookup.  Tiles whose two blocks are
// complete take a branch-free path (byte-permute decoding, one table entry
// per code decision; the LM-head State-SR, the TorchAO first moment and the
// factored v included); ragged tiles, scales outside the fast range, the
// Update-RTN and next-step rounding variants take the general one.
//
// Instantiations: step_kernel<recipe, Update-RTN, m State-SR present,
// next-step r>, with the internal recipe kRecipeFactoredOnly for launches
// whose tensors are all factored.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "q4_fastmath.cuh"
#include "q4_internal.h"
#include "q4_philox.cuh"
#include "q4_reduce.cuh"

namespace q4 {
namespace {

constexpr float kMagic = 12582912.0f;                // 1.5 * 2^23: rounds to an integer in the low mantissa bits
constexpr float kTwoM24 = 5.9604644775390625e-08f;   // 2^-24

struct __align__(16) Stage {
    uint4 grad[32];     // 256 BF16 gradients
    float4 param[64];   // 256 FP32 master weights
    uint32_t mc[32];    // m code words of both blocks (64 bytes each)
    uint32_t vc[32];    // v code words of both blocks
    float ms[2];        // m scales of both blocks
    float vs[2];        // v scales of both blocks
};
static_assert(sizeof(Stage) % 16 == 0, "stage buffers must keep 16-byte alignment");

// Per-warp tables.  256-byte aligned: the fast decoder forms the address of
// deqm/deqv entries by replacing the low byte of the table's address with
// 4*code + 64*half (+128 for v).
struct __align__(256) WarpTables {
    float deqm[32];        // [half][16] NF4 level * old s_m
    float deqv[32];        // [half][16] v level * old s_v
    float mt[2][48];       // fast path, per half: m State-SR a_{c+1} by cell (floats 0..15) and (a_k, d_k)
                           // by cell (float2 8..23); TorchAO: floats 0..8 = SDyn4 magnitudes A_0..A_7 * new
                           // s_m, +inf
    float2 rdv[2][16];     // fast path, per half: ZIP-SR (r_k, d_k) by cell
    float tm[32];          // general path: [half][16] NF4 threshold * new s_m
    float am[32];          // [half][16] NF4 level * new s_m (LM-head SR)
    float av[32];          // [half][16] v level * new s_v (ZIP-SR) or v threshold * new s_v (RTN)
    float2 rd[32];         // [half][16] (r_k, (r_k - r_{k+1}) * 2^-24) for ZIP-SR
};

constexpr int kTilesPerStage = 3;   // tiles a stage buffer holds (8 issuing lanes each)
constexpr int kStageBufs = 2;       // stage buffers per warp
static_assert(kTilesPerStage * 8 <= 32 && kStageBufs >= 2, "stage geometry");

struct __align__(256) WarpSmem {
    WarpTables wt;
    Stage st[kStageBufs][kTilesPerStage];   // stage buffers of kTilesPerStage tiles each
    DevTensor desc;                         // descriptor of the tensor being computed
    float4 rbv;                             // factored: its {mean(R), 1/mean(R), fast flag, 0}
    unsigned long long bar[kStageBufs];     // one mbarrier per stage buffer
};

struct __align__(256) SmemAll {
    WarpSmem w[kStepWarps];
    float2 nf4_bucket[64];  // NF4 RTN by linear bucket: {unscaled threshold of the candidate, candidate}
    float nf4_thr[64];      // its thresholds alone (4-byte entries: buckets 0..32 in distinct banks)
    float4 v_rtn[16];       // v RTN by candidate c: {unscaled threshold t_c, level L_c, level L_{c+1}, 0}
    float v_thr[16];        // the thresholds t_c alone: 16 words in distinct banks
    float v_next[16];       // ZIP-SR cell search by candidate c: unscaled level L_{c+1}
    float vl[16];     // unscaled v levels (EDEN reconstruction)
    uint8_t lut_nf4_t[64];
    uint8_t lut_nf4_l[64];
    uint8_t lut_v_l[kVLut];
    uint8_t lut_v_t[kVLut];
    uint8_t lut_m_log[kVLut];   // TorchAO: SDyn4 magnitude candidates
};

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity; false if it has not completed
// within `limit` SM clock cycles.  A limit below kPollBelow polls with the
// non-blocking test_wait, so that it expires even when the data would arrive
// during a try_wait suspension; longer limits suspend in try_wait between
// clock checks.  (The limit is uniform over the launch.)
constexpr long long kPollBelow = 1000000;
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity, long long limit) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (limit < kPollBelow ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}
// Predicated forms (no branch): the operation runs on lanes whose flag is set.
__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint32_t flag, uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t}" ::"r"(flag),
        "r"(bar), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_if(uint32_t flag, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%1];\n\t}" ::"r"(flag),
        "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_load_if(uint32_t flag, uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar, uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%1], [%2], %3, [%4], "
        "%5;\n\t}" ::"r"(flag),
        "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void cp_async4_if(uint32_t flag, uint32_t dst, const void* src) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p cp.async.ca.shared.global [%1], [%2], 4;\n\t}" ::"r"(flag),
        "r"(dst), "l"(src)
        : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc_if(uint32_t flag, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%1];\n\t}" ::"r"(flag),
        "r"(bar)
        : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------------------------- arithmetic helpers
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t to_bf16(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Maximum over the 16 lanes of this lane's half of a lane value x >= +0 that
// is not NaN (a max of fmaxf's started at +0).  For such floats the order of
// the bit patterns is the order of the values, so two integer warp reductions
// give the exact result.
__device__ __forceinline__ float half_max(float x, int half) {
    const uint32_t b = __float_as_uint(x);
    const uint32_t m0 = __reduce_max_sync(0xffffffffu, half ? 0u : b);
    const uint32_t m1 = __reduce_max_sync(0xffffffffu, half ? b : 0u);
    return __uint_as_float(half ? m1 : m0);
}

// Fast candidate paths need a scale whose reciprocal and scaled tables are
// normal numbers; anything else (0, subnormal, huge, NaN) takes the exact
// sequential search.
__device__ __forceinline__ bool scale_in_fast_range(float s) { return s >= 0x1p-90f && s <= 0x1p90f; }

// x >= 0 (or NaN) lies in (0, 2^-100): outside the fast square root's domain.
__device__ __forceinline__ bool tiny_positive(float x) { return (__float_as_uint(x) - 1u) < 0x0d7fffffu; }

// x >= 0 lies in {0} or [2^-100, 2^100]: the quotient's safe range.
__device__ __forceinline__ bool quot_range_ok(float x) {
    const uint32_t b = __float_as_uint(x);
    return b == 0u || (b - 0x0d800000u) <= (0x71800000u - 0x0d800000u);
}

// r = 1/(sqrt(v') c2 + eps), correctly rounded either way.
template <bool FAST>
__device__ __forceinline__ float precond(const StepParams& P, float v1) {
    if (FAST) {
        const float d = __fadd_rn(__fmul_rn(sqrt_rn_normal<0>(v1), P.c2), P.eps);
        return rcp_rn_normal<1>(d);
    }
    return __frcp_rn(__fadd_rn(__fmul_rn(__fsqrt_rn(v1), P.c2), P.eps));
}

// Next-step zero-gradient preconditioner 1/(sqrt(beta2 x) c2(t+1) + eps), the
// rounding space of the next-step ZIP-SR variant (IEEE operations only).
__device__ __forceinline__ float precond_next(const StepParams& P, float x) {
    return __frcp_rn(__fadd_rn(__fmul_rn(__fsqrt_rn(__fmul_rn(P.beta2, x)), P.c2_next), P.eps));
}

// precond_next through the correctly rounded fast square root and reciprocal
// where their domains hold (beta2 x is +0 or in [2^-100, inf), the divisor
// below 2^126; the divisor is at least eps >= 2^-100 under fast_math), else
// the IEEE operations: the same value either way.
__device__ __forceinline__ float precond_next_fast(const StepParams& P, float x) {
    const float bx = __fmul_rn(P.beta2, x);
    if (P.fast_math && sqrt_fast_domain(bx)) {
        const float d = __fadd_rn(__fmul_rn(sqrt_rn_normal<0>(bx), P.c2_next), P.eps);
        if (d < 0x1p126f) return rcp_rn_normal<1>(d);
    }
    return precond_next(P, x);
}

// The same on a pair.
__device__ __forceinline__ float2 precond_next_fast2(const StepParams& P, float2 x) {
    const float2 bx = mul2_rn(P.x2_beta2, x);
    if (P.fast_math && sqrt_fast_domain(bx.x) && sqrt_fast_domain(bx.y)) {
        // the paired product feeds scalar adds only
        const float2 sc = mul2_rn(sqrt2_rn_normal(bx), make_float2(P.c2_next, P.c2_next));
        const float2 d = make_float2(__fadd_rn(sc.x, P.eps), __fadd_rn(sc.y, P.eps));
        if (d.x < 0x1p126f && d.y < 0x1p126f) return rcp2_rn_normal(d);
    }
    return make_float2(precond_next(P, x.x), precond_next(P, x.y));
}

// The update of 8 elements: r_i and theta'_i.
template <bool FAST>
__device__ __forceinline__ void update8(const StepParams& P, const float m1[8], const float v1[8], float th[8],
                                        float r[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        r[i] = precond<FAST>(P, v1[i]);
        th[i] = __fsub_rn(__fmul_rn(th[i], P.decay), __fmul_rn(P.step_size, __fmul_rn(m1[i], r[i])));
    }
}

// ----------------------------------------------------------------- paired arithmetic
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

// Moments and update of the lane's 8 elements as 4 pairs (2k, 2k+1), with the
// paired FP32 instructions; each component rounds as the scalar sequence:
// m' = fma(b1, m, omb1 g), v' = fma(b2, v, omb2 (g g)),
// r = 1/(sqrt(v') c2 + eps), theta' = theta decay + (-step) (m' r), where
// theta decay - step (m' r) = theta decay + (-step) (m' r) exactly.
// Lanes with a v' outside the fast square root's domain take the scalar IEEE
// sequence.
__device__ __forceinline__ float update_pairs(const StepParams& P, const float2 g[4], const float2 m[4],
                                              const float2 v[4], bool fact, float2 m1[4], float2 v1[4],
                                              float2 th[4], float2 r[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        m1[k] = fma2_rn(P.x2_beta1, m[k], mul2_rn(P.x2_omb1, g[k]));
        if (!fact) v1[k] = fma2_rn(P.x2_beta2, v[k], mul2_rn(P.x2_omb2, mul2_rn(g[k], g[k])));
    }
    // lane max of v' (the block scale input) and min (the fast square root's
    // domain: every v' is +0 or in [2^-100, +inf))
    float vmax = 0.f, vmin = INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        vmax = fmaxf(vmax, fmaxf(v1[k].x, v1[k].y));
        vmin = fminf(vmin, fminf(v1[k].x, v1[k].y));
    }
    bool tiny = false;
    if (!(vmin >= 0x1p-100f)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) tiny = tiny || tiny_positive(v1[k].x) || tiny_positive(v1[k].y);
    }
    if (P.fast_math && !tiny && vmax < INFINITY) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // products paired, sums scalar (a paired product must not feed a paired add)
            const float2 sc = mul2_rn(sqrt2_rn_normal(v1[k]), P.x2_c2);
            r[k] = rcp2_rn_normal(make_float2(__fadd_rn(sc.x, P.eps), __fadd_rn(sc.y, P.eps)));
            const float2 t1 = mul2_rn(th[k], P.x2_decay);
            const float2 t2 = mul2_rn(P.x2_neg_step, mul2_rn(m1[k], r[k]));
            th[k] = make_float2(__fadd_rn(t1.x, t2.x), __fadd_rn(t1.y, t2.y));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r[k].x = precond<false>(P, v1[k].x);
            r[k].y = precond<false>(P, v1[k].y);
            th[k].x = __fsub_rn(__fmul_rn(th[k].x, P.decay), __fmul_rn(P.step_size, __fmul_rn(m1[k].x, r[k].x)));
            th[k].y = __fsub_rn(__fmul_rn(th[k].y, P.decay), __fmul_rn(P.step_size, __fmul_rn(m1[k].y, r[k].y)));
        }
    }
    return vmax;
}

// Packs eight 4-bit codes (element i in bits 4i..4i+3) with a shallow tree.
__device__ __forceinline__ uint32_t pack8(const uint32_t c[8]) {
    const uint32_t b0 = c[0] + (c[1] << 4), b1 = c[2] + (c[3] << 4);
    const uint32_t b2 = c[4] + (c[5] << 4), b3 = c[6] + (c[7] << 4);
    return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// ----------------------------------------------------------------- requantisation, general path
// Codes and scales of a tile from the updated moments m1, v1 (elements beyond
// numel already zeroed), the new scales s_m, s_v and r (ZIP-SR).  Handles
// every case: partial blocks, LM-head stochastic rounding, scales outside the
// fast range (exact sequential searches).
template <int RECIPE, bool URTN, bool NEXTR>
__device__ __forceinline__ void requant_general(const StepParams& P, const DevTensor& d, const SmemAll& sm,
                                                WarpTables& wt, int lane, int64_t blk, bool blk_ok, int64_t e0,
                                                int nvalid, bool fact, bool m_sr, const float m1[8],
                                                const float v1[8], const float r[8], float s_m, float s_v,
                                                float my_nf4, float my_nf4t, float my_vl, float my_vt) {
    const int half = lane >> 4, j = lane & 15, hb = half * 16;
    wt.tm[hb + j] = __fmul_rn(my_nf4t, s_m);
    if (m_sr) wt.am[hb + j] = __fmul_rn(my_nf4, s_m);
    if (RECIPE == Q4_RECIPE_ZIP_SR) {
        const float a = __fmul_rn(my_vl, s_v);
        const float rk = NEXTR ? precond_next(P, a)
                               : (P.fast_math && scale_in_fast_range(s_v)) ? precond<true>(P, a) : precond<false>(P, a);
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
        const bool in_range = scale_in_fast_range(s_m);
        // linear-bucket candidate tables: NF4 only (the TorchAO SDyn4 map has
        // several thresholds per bucket near zero)
        const bool fast = in_range && RECIPE != Q4_RECIPE_TORCHAO;
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
                } else if (RECIPE == Q4_RECIPE_TORCHAO && in_range) {
                    // #{k : x > T_k} by binary search over the ascending scaled
                    // thresholds (normal scale: T_k is non-decreasing in k)
                    int pos = (x > wt.tm[hb + 7]) ? 8 : 0;
                    pos += (x > wt.tm[hb + pos + 3]) ? 4 : 0;
                    pos += (x > wt.tm[hb + pos + 1]) ? 2 : 0;
                    pos += (x > wt.tm[hb + pos]) ? 1 : 0;
                    code = pos;
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
            if (!URTN) draws8(d.elem_offset + (uint64_t)e0, 1u, d.tensor_id, P.step, P.round_keys, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = v1[i];
                int k;
                if (fast) {
                    const uint32_t bi = __float_as_uint(__fmul_rn(fabsf(x), rho)) >> 19;
                    const int c = sm.lut_v_l[bi];
                    k = c + (wt.av[hb + c + 1] <= x ? 1 : 0);
                } else {
                    k = 0;
#pragma unroll 1
                    for (int q = 0; q < 16; ++q)
                        if (wt.av[hb + q] <= x) k = q;
                }
                const float2 e = wt.rd[hb + k];
                // the r being rounded: the update's, or the next step's
                const float ri = NEXTR ? precond_next(P, x) : r[i];
                int code;
                if (URTN) {
                    // Update-RTN: the neighbour whose preconditioner is nearer
                    // to r (a tie keeps k)
                    code = k == 15 ? 15 : k + (__fsub_rn(ri, wt.rd[hb + k + 1].x) < __fsub_rn(e.x, ri) ? 1 : 0);
                } else {
                    // u * (r_k - r_{k+1}) with u = (w >> 8) 2^-24, as (w >> 8) * ((r_k - r_{k+1}) 2^-24)
                    code = k + (__fmul_rn((float)(w[i] >> 8), e.y) < __fsub_rn(e.x, ri) ? 1 : 0);
                }
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
                    const uint32_t bi = __float_as_uint(__fmul_rn(fabsf(x), rho)) >> 19;
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
}

// ----------------------------------------------------------------- factored second moment
// vhat = R_i * C_j / mean(R) for the lane's 8 elements; mean(R) and its
// correctly rounded reciprocal come from the statistics pass.
__device__ __forceinline__ void factored_vhat(const DevTensor& d, int64_t e0, int nvalid, float v1[8]) {
    const float2 rb = *reinterpret_cast<const float2*>(d.rbar);
    const bool rb_ok = rb.x != 0.f && quot_range_ok(rb.x);
    float R[8], C[8];
    const int64_t me0 = d.fbase + e0;   // matrix index of the lane's first element
    if (nvalid == 8 && (d.flags & DF_CVEC)) {
        const int64_t frow = me0 / d.cols;
        const int64_t fcol = me0 - frow * d.cols;
        const float Ri = __ldg(d.vrow + frow);
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(d.vcol + fcol));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(d.vcol + fcol + 4));
        C[0] = c0.x; C[1] = c0.y; C[2] = c0.z; C[3] = c0.w;
        C[4] = c1.x; C[5] = c1.y; C[6] = c1.z; C[7] = c1.w;
#pragma unroll
        for (int i = 0; i < 8; ++i) R[i] = Ri;
    } else {
        int64_t frow = 0, fcol = 0;
        if (nvalid > 0) {
            frow = me0 / d.cols;
            fcol = me0 - frow * d.cols;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            R[i] = 0.f;
            C[i] = 0.f;
            if (i < nvalid) {
                R[i] = __ldg(d.vrow + frow);
                C[i] = __ldg(d.vcol + fcol);
                if (++fcol == d.cols) { fcol = 0; ++frow; }
            }
        }
    }
    bool q_fast = rb_ok;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float p = __fmul_rn(R[i], C[i]);
        const float q = div_rn_by_rcp(p, rb.x, rb.y);
        q_fast = q_fast && quot_range_ok(p) && quot_range_ok(q);
        v1[i] = (rb.x == 0.f) ? 0.f : q;
    }
    if (!q_fast) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v1[i] = (rb.x == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(R[i], C[i]), rb.x);
    }
}

// Update of the lane's elements from m, v (dequantised) and g: moments,
// preconditioner, weights.  Returns whether the fast square root/reciprocal
// were used (irrelevant to the results, which are identical either way).
__device__ __forceinline__ void moments_and_update(const StepParams& P, const float g[8], const float m[8],
                                                   const float v[8], bool fact, float m1[8], float v1[8],
                                                   float th[8], float r[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m1[i] = __fmaf_rn(P.beta1, m[i], __fmul_rn(P.omb1, g[i]));
        if (!fact) v1[i] = __fmaf_rn(P.beta2, v[i], __fmul_rn(P.omb2, __fmul_rn(g[i], g[i])));
    }
    bool tiny = false;
    float vmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        tiny = tiny || tiny_positive(v1[i]);
        vmax = fmaxf(vmax, v1[i]);
    }
    if (P.fast_math && !tiny && vmax < INFINITY) update8<true>(P, m1, v1, th, r);
    else update8<false>(P, m1, v1, th, r);
}

// vhat for 8 elements of one row from preloaded R_i, C_j (8 columns) and
// {mean(R), RN(1/mean(R))}: p = R_i C_j and q = p / mean(R) with the paired
// quotient, the same operations and fallback as factored_vhat.  The quotient
// is exact when every p and q is 0 or in [2^-100, 2^100]; as R_i, C_j >= 0 and
// both roundings are monotone, that follows from the largest C_j and the
// smallest nonzero one (the q bounds are taken with a factor-2 margin, as the
// bounds themselves come from the fast quotient).
__device__ __forceinline__ void factored_vhat_pre(const float Ri, const float4 c0, const float4 c1, const float2 rb,
                                                  float v1[8]) {
    const float C[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    // on the bit patterns of the non-negative C_j: the largest (NaN and +inf
    // above every finite value) and the smallest nonzero (minus 1; all ones: none)
    uint32_t cmax_b = 0u, cmin_m1 = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cmax_b = max(cmax_b, __float_as_uint(C[i]));
        cmin_m1 = min(cmin_m1, __float_as_uint(C[i]) - 1u);
    }
    bool q_fast = rb.x != 0.f && quot_range_ok(rb.x);
    if (Ri != 0.f && cmin_m1 != 0xffffffffu) {
        const float pmax = __fmul_rn(Ri, __uint_as_float(cmax_b));
        const float pmin = __fmul_rn(Ri, __uint_as_float(cmin_m1 + 1u));
        q_fast = q_fast && quot_range_ok(pmax) && quot_range_ok(pmin);
        if (q_fast) {
            const float2 qb = div2_rn_by_rcp(make_float2(pmin, pmax), rb.x, rb.y);
            q_fast = qb.x >= 0x1p-99f && qb.y <= 0x1p99f;
        }
    }
    if (q_fast) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 p = mul2_rn(make_float2(Ri, Ri), make_float2(C[2 * k], C[2 * k + 1]));
            const float2 q = div2_rn_by_rcp(p, rb.x, rb.y);
            v1[2 * k] = q.x;
            v1[2 * k + 1] = q.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v1[i] = (rb.x == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(Ri, C[i]), rb.x);
    }
}

// ----------------------------------------------------------------- one tile, general path
// `st` is the staged tile or nullptr (ragged tail: read from global memory).
template <int RECIPE, bool URTN, bool NEXTR>
__device__ __forceinline__ void compute_tile(const StepParams& P, const DevTensor& d, int64_t pair,
                                             const Stage* st, int lane, SmemAll& sm, WarpTables& wt,
                                             const float my_nf4, const float my_nf4t, const float my_vl,
                                             const float my_vt, const float clip) {
    const int half = lane >> 4, j = lane & 15, hb = half * 16;
    const int64_t numel = d.numel;
    const int64_t nblk = (numel + kBlock - 1) / kBlock;
    const int64_t blk = pair * 2 + half;
    const bool blk_ok = blk < nblk;
    const int64_t e0 = blk * kBlock + j * 8;
    const int64_t rem = numel - e0;
    const int nvalid = rem >= 8 ? 8 : (rem > 0 ? (int)rem : 0);
    const uint32_t flags = d.flags;
    const bool fact = is_factored_recipe(RECIPE) && (RECIPE == kRecipeFactoredOnly || (flags & DF_FACTORED));
    const bool m_sr = (flags & DF_M_SR) != 0;

    // ---- loads -------------------------------------------------------
    float g[8], th[8];
    uint32_t qmw = 0, qvw = 0;
    float sm_old = 0.f, sv_old = 0.f;
    if (st != nullptr) {
        if (blk_ok) {
            sm_old = st->ms[half];
            qmw = st->mc[hb + j];
            if (!fact) {
                sv_old = st->vs[half];
                qvw = st->vc[hb + j];
            }
        }
        if (nvalid == 8) {
            const uint4 gw = st->grad[hb + j];
            const float4 t0 = st->param[2 * (hb + j)];
            const float4 t1 = st->param[2 * (hb + j) + 1];
            g[0] = bf16lo(gw.x); g[1] = bf16hi(gw.x); g[2] = bf16lo(gw.y); g[3] = bf16hi(gw.y);
            g[4] = bf16lo(gw.z); g[5] = bf16hi(gw.z); g[6] = bf16lo(gw.w); g[7] = bf16hi(gw.w);
            th[0] = t0.x; th[1] = t0.y; th[2] = t0.z; th[3] = t0.w;
            th[4] = t1.x; th[5] = t1.y; th[6] = t1.z; th[7] = t1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) g[i] = th[i] = 0.f;
        }
    } else {
        if (blk_ok) {
            sm_old = __ldg(d.ms + blk);
            qmw = __ldg(reinterpret_cast<const uint32_t*>(d.mc + blk * 64) + j);
            if (!fact) {
                sv_old = __ldg(d.vs + blk);
                qvw = __ldg(reinterpret_cast<const uint32_t*>(d.vc + blk * 64) + j);
            }
        }
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

    // global-norm clipping scales the FP32 gradient first (1 when off)
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = __fmul_rn(g[i], clip);

    // ---- dequantisation (old scales) and update --------------------------
    wt.deqm[hb + j] = __fmul_rn(my_nf4, sm_old);
    if (!fact) wt.deqv[hb + j] = __fmul_rn(my_vl, sv_old);
    __syncwarp();
    float m[8], v[8], m1[8], v1[8], r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m[i] = wt.deqm[hb + ((qmw >> (4 * i)) & 15u)];
        v[i] = fact ? 0.f : wt.deqv[hb + ((qvw >> (4 * i)) & 15u)];
    }
    if (fact) factored_vhat(d, e0, nvalid, v1);
    moments_and_update(P, g, m, v, fact, m1, v1, th, r);
    float amax = 0.f, vmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i >= nvalid) { m1[i] = 0.f; v1[i] = 0.f; }
        amax = fmaxf(amax, fabsf(m1[i]));
        vmax = fmaxf(vmax, v1[i]);
    }

    // ---- weights out ----------------------------------------------------
    if (nvalid == 8) {
        __stcs(reinterpret_cast<float4*>(d.param + e0), make_float4(th[0], th[1], th[2], th[3]));
        __stcs(reinterpret_cast<float4*>(d.param + e0 + 4), make_float4(th[4], th[5], th[6], th[7]));
        if (flags & DF_BF16) {
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
                if (flags & DF_BF16) d.bf16[e0 + i] = to_bf16(th[i]);
            }
        }
    }

    const float s_m = half_max(amax, half);
    const float s_v = fact ? 0.f : half_max(vmax, half);
    requant_general<RECIPE, URTN, NEXTR>(P, d, sm, wt, lane, blk, blk_ok, e0, nvalid, fact, m_sr, m1, v1, r, s_m, s_v,
                                  my_nf4, my_nf4t, my_vl, my_vt);
}

// ----------------------------------------------------------------- one tile, fast path
// A staged tile whose two blocks are both complete (256 elements).  Decoding
// reads the dequantisation tables through addresses built with byte permutes;
// when neither block needs the general requantisation (LM-head stochastic
// rounding, or a new scale outside the fast range) the codes come from
// per-bucket entries that carry everything one comparison needs.
template <int RECIPE, bool URTN, bool MSR, bool NEXTR>
__device__ __forceinline__ void compute_tile_full(const StepParams& P, const DevTensor& d, int64_t pair,
                                                  const Stage& st, int lane, SmemAll& sm, WarpTables& wt,
                                                  const float my_nf4, const float my_nf4t, const float my_vl,
                                                  const float my_vt, const float my_vl1, const float my_mag,
                                                  const float clip, const uint32_t f_row, const uint32_t f_col,
                                                  const float4& rbv) {
    const int half = lane >> 4, j = lane & 15, hb = half * 16;
    const int64_t blk = pair * 2 + half;
    const int64_t e0 = blk * kBlock + j * 8;
    const uint32_t flags = d.flags;
    const bool fact = is_factored_recipe(RECIPE) && (RECIPE == kRecipeFactoredOnly || (flags & DF_FACTORED));
    const bool m_sr = (flags & DF_M_SR) != 0;
    const uint32_t tb = smem_addr(&wt);   // 256-byte aligned

    // factored v with columns a multiple of 8, at least 256: the tile starts at
    // (f_row, f_col) and the lane's 8 elements lie in one row
    const bool fvec = fact && (flags & DF_CVEC);

    // ---- loads from the stage ---------------------------------------------
    const float sm_old = st.ms[half];
    const uint32_t qmw = st.mc[hb + j];
    const float sv_old = fact ? 0.f : st.vs[half];
    const uint32_t qvw = fact ? 0u : st.vc[hb + j];
    float2 g[4], th[4];
    {
        const uint4 gw = st.grad[hb + j];
        const float4 t0 = st.param[2 * (hb + j)];
        const float4 t1 = st.param[2 * (hb + j) + 1];
        g[0] = make_float2(bf16lo(gw.x), bf16hi(gw.x));
        g[1] = make_float2(bf16lo(gw.y), bf16hi(gw.y));
        g[2] = make_float2(bf16lo(gw.z), bf16hi(gw.z));
        g[3] = make_float2(bf16lo(gw.w), bf16hi(gw.w));
        const float2 clip2 = make_float2(clip, clip);   // global-norm clipping (1 when off)
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = mul2_rn(g[k], clip2);
        th[0] = make_float2(t0.x, t0.y);
        th[1] = make_float2(t0.z, t0.w);
        th[2] = make_float2(t1.x, t1.y);
        th[3] = make_float2(t1.z, t1.w);
    }

    // ---- dequantisation: table entry address = table | (4 code + 64 half [+ 128 for v])
    wt.deqm[hb + j] = __fmul_rn(my_nf4, sm_old);
    if (!fact) wt.deqv[hb + j] = __fmul_rn(my_vl, sv_old);
    __syncwarp();
    float2 m[4], v[4], m1[4], v1[4], r[4];
    {
        const uint32_t hbytes = half ? 0x40404040u : 0u;
        const uint32_t mlo = ((qmw << 2) & 0x3C3C3C3Cu) | hbytes;
        const uint32_t mhi = ((qmw >> 2) & 0x3C3C3C3Cu) | hbytes;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[k] = make_float2(lds_f32(__byte_perm(mlo, tb, 0x7650 + k)), lds_f32(__byte_perm(mhi, tb, 0x7650 + k)));
        if (!fact) {
            const uint32_t vlo = ((qvw << 2) & 0x3C3C3C3Cu) | hbytes | 0x80808080u;
            const uint32_t vhi = ((qvw >> 2) & 0x3C3C3C3Cu) | hbytes | 0x80808080u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[k] = make_float2(lds_f32(__byte_perm(vlo, tb, 0x7650 + k)),
                                   lds_f32(__byte_perm(vhi, tb, 0x7650 + k)));
        } else {
            float vf[8];
            // R_i, the lane's 8 C_j and mean(R), loaded where the quotient
            // needs them (loads at the tile's start, for more overlap, measured
            // slower: longer live ranges)
            float f_ri = 0.f;
            float4 f_c0 = make_float4(0.f, 0.f, 0.f, 0.f), f_c1 = f_c0;
            float2 f_rb = make_float2(0.f, 0.f);
            bool f_fast = false;   // every quotient of the tensor in the fast quotient's exact range
            if (is_factored_recipe(RECIPE) && fvec) {
                const uint32_t cols = (uint32_t)d.cols;
                uint32_t col = f_col + (uint32_t)(half * kBlock + j * 8), row = f_row;
                if (col >= cols) { col -= cols; ++row; }
                f_ri = __ldg(d.vrow + row);
                f_c0 = __ldg(reinterpret_cast<const float4*>(d.vcol + col));
                f_c1 = __ldg(reinterpret_cast<const float4*>(d.vcol + col + 4));
                const float4 rb4 = rbv;
                f_rb = make_float2(rb4.x, rb4.y);
                f_fast = rb4.z != 0.f;
            }
            if (fvec && f_fast) {
                const float C[8] = {f_c0.x, f_c0.y, f_c0.z, f_c0.w, f_c1.x, f_c1.y, f_c1.z, f_c1.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 p = mul2_rn(make_float2(f_ri, f_ri), make_float2(C[2 * k], C[2 * k + 1]));
                    const float2 q = div2_rn_by_rcp(p, f_rb.x, f_rb.y);
                    vf[2 * k] = q.x;
                    vf[2 * k + 1] = q.y;
                }
            } else if (fvec) {
                factored_vhat_pre(f_ri, f_c0, f_c1, f_rb, vf);
            } else {
                factored_vhat(d, e0, 8, vf);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[k] = make_float2(0.f, 0.f);
                v1[k] = make_float2(vf[2 * k], vf[2 * k + 1]);
            }
        }
    }
    const float vmax_lane = update_pairs(P, g, m, v, fact, m1, v1, th, r);

    // ---- weights out ----------------------------------------------------
    __stcs(reinterpret_cast<float4*>(d.param + e0), make_float4(th[0].x, th[0].y, th[1].x, th[1].y));
    __stcs(reinterpret_cast<float4*>(d.param + e0 + 4), make_float4(th[2].x, th[2].y, th[3].x, th[3].y));
    if (flags & DF_BF16) {
        uint4 o;
        o.x = pack_bf16x2(th[0].x, th[0].y);
        o.y = pack_bf16x2(th[1].x, th[1].y);
        o.z = pack_bf16x2(th[2].x, th[2].y);
        o.w = pack_bf16x2(th[3].x, th[3].y);
        __stcs(reinterpret_cast<uint4*>(d.bf16 + e0), o);
    }

    // ---- block scales -----------------------------------------------------
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(m1[k].x), fabsf(m1[k].y)));
    const float s_m = half_max(amax, half);
    const float s_v = fact ? 0.f : half_max(vmax_lane, half);

    const bool fast = __all_sync(0xffffffffu, (MSR || !m_sr) && scale_in_fast_range(s_m) &&
                                                          (fact || scale_in_fast_range(s_v)));
    if (!fast) {
        float m1s[8], v1s[8], rs[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m1s[2 * k] = m1[k].x; m1s[2 * k + 1] = m1[k].y;
            v1s[2 * k] = v1[k].x; v1s[2 * k + 1] = v1[k].y;
            rs[2 * k] = r[k].x; rs[2 * k + 1] = r[k].y;
        }
        requant_general<RECIPE, URTN, false>(P, d, sm, wt, lane, blk, true, e0, 8, fact, m_sr, m1s, v1s, rs, s_m, s_v,
                                      my_nf4, my_nf4t, my_vl, my_vt);
        return;
    }

    // ---- m codes, NF4 RTN: no per-block table ------------------------------
    // The linear bucket b of m' (buckets 0..32 occur for |m'| <= s_m) reads
    // the CTA's constant entry {t_c, c} (c the candidate code, t_c its
    // unscaled threshold); the threshold at the new scale is t_c * s_m, the
    // same product a per-block table would hold.  Computed ahead of the table
    // stores below so that it overlaps their dependency chain.
    const bool nf4_rtn = RECIPE != Q4_RECIPE_TORCHAO && !(MSR && m_sr);
    uint32_t cm = 0;
    if (nf4_rtn) {
        const float rho16 = __fmul_rn(16.f, rcp_rn_normal<1>(s_m));
        const uint32_t nb_base = smem_addr(sm.nf4_bucket);
        const uint32_t nt_base = smem_addr(sm.nf4_thr), nc_base = smem_addr(sm.lut_nf4_t);
        const float2 sm2 = make_float2(s_m, s_m);
        uint32_t c[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 z = fma2_rn(m1[k], make_float2(rho16, rho16), make_float2(kMagic + 16.f, kMagic + 16.f));
            const uint32_t b0 = __float_as_uint(z.x) & 63u, b1 = __float_as_uint(z.y) & 63u;
            float2 thr;
            uint32_t q0, q1;
            if (RECIPE == Q4_RECIPE_ZE_EDEN) {
                // two 4-byte reads, free of bank conflicts (measured faster here;
                // one 8-byte read of {t_c, c} is faster for ZIP-SR)
                thr = make_float2(lds_f32(nt_base + b0 * 4u), lds_f32(nt_base + b1 * 4u));
                q0 = lds_u8(nc_base + b0);
                q1 = lds_u8(nc_base + b1);
            } else {
                const float2 e0v = lds_f32x2(nb_base + b0 * 8u), e1v = lds_f32x2(nb_base + b1 * 8u);
                thr = make_float2(e0v.x, e1v.x);
                q0 = __float_as_uint(e0v.y);
                q1 = __float_as_uint(e1v.y);
            }
            thr = mul2_rn(thr, sm2);
            c[2 * k] = q0 + (m1[k].x > thr.x ? 1u : 0u);
            c[2 * k + 1] = q1 + (m1[k].y > thr.y ? 1u : 0u);
        }
        cm = pack8(c);
    }

    // ---- fast tables at the new scales ------------------------------------
    // State-SR (LM head during its SR phase): a_k = level k at the new scale;
    // the cell search reads a_{c+1} (floats 0..15 of mt[half]), then
    // (a_k, d_k) with d_k = (a_{k+1} - a_k) 2^-24 (float2 8..23).
    if (RECIPE == Q4_RECIPE_TORCHAO) {
        reinterpret_cast<float*>(&wt.mt[half][0])[j] = __fmul_rn(my_mag, s_m);   // A_j s_m; +inf from j = 8
    } else if (MSR && m_sr) {
        const float a = __fmul_rn(my_nf4, s_m);
        const float a1 = __shfl_down_sync(0xffffffffu, a, 1);
        float* mb = reinterpret_cast<float*>(&wt.mt[half][0]);
        mb[j] = a1;
        reinterpret_cast<float2*>(mb + 16)[j] = make_float2(a, j < 15 ? __fmul_rn(__fsub_rn(a1, a), kTwoM24) : 0.f);
    }
    if (RECIPE == Q4_RECIPE_ZIP_SR && !fact) {
        // a_k = level k at the new scale, r_k its preconditioner, d_k =
        // (r_k - r_{k+1}) 2^-24: after the cell search (from the constant
        // levels) the SR decision reads (r_k, d_k) by cell; Update-RTN reads
        // (r_k, r_{k+1}) instead (r_15 twice: cell 15 keeps code 15).
        const float a = __fmul_rn(my_vl, s_v);
        const float rk = NEXTR ? precond_next_fast(P, a) : P.fast_math ? precond<true>(P, a) : precond<false>(P, a);
        const float rk1 = __shfl_down_sync(0xffffffffu, rk, 1);
        const float dk = URTN ? (j < 15 ? rk1 : rk) : j < 15 ? __fmul_rn(__fsub_rn(rk, rk1), kTwoM24) : 0.f;
        wt.rdv[half][j] = make_float2(rk, dk);
    }
    // the v RTN codes (ZE-EDEN, TorchAO, factored 1-D) and the NF4 RTN m codes
    // read constant tables only: no per-block table to wait for
    if (RECIPE == Q4_RECIPE_ZIP_SR || RECIPE == Q4_RECIPE_TORCHAO || (MSR && m_sr)) __syncwarp();

    // ---- m codes: NF4 State-SR; TorchAO SDyn4 RTN by magnitude ----------------
    if (RECIPE == Q4_RECIPE_TORCHAO) {
        // count n = #{i : A_i s_m below |m'|} from the log-bucket lower bound c
        // and one comparison with A_c s_m (strict for m' >= 0, non-strict for
        // m' < 0); code = 7 + n, or 7 - min(n, 7) for m' < 0
        const float rho = rcp_rn_normal<1>(s_m);
        const uint32_t mt_base = tb + (uint32_t)((char*)&wt.mt[half][0] - (char*)&wt);
        const uint32_t lut = smem_addr(sm.lut_m_log);
        uint32_t c[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 ax = make_float2(fabsf(m1[k].x), fabsf(m1[k].y));
            const float2 y = mul2_rn(ax, make_float2(rho, rho));
            const uint32_t c0 = lds_u8(lut + (__float_as_uint(y.x) >> 19));
            const uint32_t c1 = lds_u8(lut + (__float_as_uint(y.y) >> 19));
            const float a0 = lds_f32(mt_base + c0 * 4u), a1 = lds_f32(mt_base + c1 * 4u);
            const bool neg0 = m1[k].x < 0.f, neg1 = m1[k].y < 0.f;
            const uint32_t n0 = c0 + ((neg0 ? ax.x >= a0 : ax.x > a0) ? 1u : 0u);
            const uint32_t n1 = c1 + ((neg1 ? ax.y >= a1 : ax.y > a1) ? 1u : 0u);
            c[2 * k] = neg0 ? 7u - min(n0, 7u) : 7u + n0;
            c[2 * k + 1] = neg1 ? 7u - min(n1, 7u) : 7u + n1;
        }
        cm = pack8(c);
    } else if (MSR && m_sr) {
        const float rho16 = __fmul_rn(16.f, rcp_rn_normal<1>(s_m));
        const uint32_t mt_base = tb + (uint32_t)((char*)&wt.mt[half][0] - (char*)&wt);
        const uint32_t lut = smem_addr(sm.lut_nf4_l);
        uint32_t w[8], c[8];
        draws8(d.elem_offset + (uint64_t)e0, 0u, d.tensor_id, P.step, P.round_keys, w);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 z = fma2_rn(m1[k], make_float2(rho16, rho16), make_float2(kMagic + 16.f, kMagic + 16.f));
            const uint32_t c0 = lds_u8(lut + (__float_as_uint(z.x) & 63u));
            const uint32_t c1 = lds_u8(lut + (__float_as_uint(z.y) & 63u));
            const uint32_t k0 = c0 + (lds_f32(mt_base + c0 * 4u) <= m1[k].x ? 1u : 0u);
            const uint32_t k1 = c1 + (lds_f32(mt_base + c1 * 4u) <= m1[k].y ? 1u : 0u);
            const float2 e0v = lds_f32x2(mt_base + 64u + k0 * 8u);
            const float2 e1v = lds_f32x2(mt_base + 64u + k1 * 8u);
            // u (a_{k+1} - a_k) with u = (w >> 8) 2^-24, as (w >> 8) ((a_{k+1} - a_k) 2^-24)
            const float2 t = mul2_rn(make_float2((float)(w[2 * k] >> 8), (float)(w[2 * k + 1] >> 8)),
                                     make_float2(e0v.y, e1v.y));
            const float2 gap = add2_rn(m1[k], make_float2(-e0v.x, -e1v.x));
            c[2 * k] = k0 + (t.x < gap.x ? 1u : 0u);
            c[2 * k + 1] = k1 + (t.y < gap.y ? 1u : 0u);
        }
        cm = pack8(c);
    }

    // ---- v codes ----------------------------------------------------------
    uint32_t cv = 0;
    float sv_store = s_v;
    if (!fact) {
        const float rho = rcp_rn_normal<1>(s_v);
        const uint32_t rd_base = tb + (uint32_t)((char*)&wt.rdv[half][0] - (char*)&wt);
        uint32_t c[8];
        const float2 sv2 = make_float2(s_v, s_v);
        if (RECIPE == Q4_RECIPE_ZIP_SR) {
            const uint32_t lut = smem_addr(sm.lut_v_l);
            const uint32_t vn_base = smem_addr(sm.v_next);
            uint32_t w[8];
            if (!URTN) draws8(d.elem_offset + (uint64_t)e0, 1u, d.tensor_id, P.step, P.round_keys, w);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 y = mul2_rn(v1[k], make_float2(rho, rho));
                const uint32_t c0 = lds_u8(lut + (__float_as_uint(y.x) >> 19));
                const uint32_t c1 = lds_u8(lut + (__float_as_uint(y.y) >> 19));
                // a_{c+1} = L_{c+1} * s_v, the level at the new scale
                const float2 a1 = mul2_rn(make_float2(lds_f32(vn_base + c0 * 4u), lds_f32(vn_base + c1 * 4u)), sv2);
                const bool up0 = a1.x <= v1[k].x;
                const bool up1 = a1.y <= v1[k].y;
                const uint32_t k0 = c0 + (up0 ? 1u : 0u), k1 = c1 + (up1 ? 1u : 0u);
                const float2 e0v = lds_f32x2(rd_base + k0 * 8u);
                const float2 e1v = lds_f32x2(rd_base + k1 * 8u);
                const float2 rk = make_float2(e0v.x, e1v.x);
                const float2 dk = make_float2(e0v.y, e1v.y);
                // the r being rounded: the update's, or the next step's
                const float2 ri = NEXTR ? precond_next_fast2(P, v1[k]) : r[k];
                const float2 gap = add2_rn(rk, neg2(ri));
                if (URTN) {
                    // Update-RTN: up when r - r_{k+1} < r_k - r (a tie keeps k)
                    const float2 below = add2_rn(ri, neg2(dk));
                    c[2 * k] = k0 + (below.x < gap.x ? 1u : 0u);
                    c[2 * k + 1] = k1 + (below.y < gap.y ? 1u : 0u);
                } else {
                    // u (r_k - r_{k+1}) with u = (w >> 8) 2^-24, as (w >> 8) ((r_k - r_{k+1}) 2^-24)
                    const float2 t = mul2_rn(make_float2((float)(w[2 * k] >> 8), (float)(w[2 * k + 1] >> 8)), dk);
                    c[2 * k] = k0 + (t.x < gap.x ? 1u : 0u);
                    c[2 * k + 1] = k1 + (t.y < gap.y ? 1u : 0u);
                }
            }
        } else {
            const uint32_t lut = smem_addr(sm.lut_v_t);
            const uint32_t vr_base = smem_addr(sm.v_rtn);
            const uint32_t vt_base = smem_addr(sm.v_thr);
            const uint32_t vl_base = smem_addr(sm.vl);
            // EDEN: each group of 4 consecutive elements (pairs 2h, 2h+1)
            // summed left to right as its terms appear
            float pa[2] = {0.f, 0.f}, pb[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 y = mul2_rn(v1[k], make_float2(rho, rho));
                const uint32_t c0 = lds_u8(lut + (__float_as_uint(y.x) >> 19));
                const uint32_t c1 = lds_u8(lut + (__float_as_uint(y.y) >> 19));
                // the threshold at the new scale is t_c * s_v; TorchAO reads it from
                // the {t_c, L_c, L_{c+1}} entry, ZE-EDEN from the 4-byte table (no
                // bank conflicts) and then the level of the chosen code
                float2 thr;
                if (RECIPE == Q4_RECIPE_ZE_EDEN) {
                    thr = make_float2(lds_f32(vt_base + c0 * 4u), lds_f32(vt_base + c1 * 4u));
                } else {
                    thr = make_float2(lds_f32x4(vr_base + c0 * 16u).x, lds_f32x4(vr_base + c1 * 16u).x);
                }
                thr = mul2_rn(thr, sv2);
                const bool up0 = v1[k].x > thr.x, up1 = v1[k].y > thr.y;
                c[2 * k] = c0 + (up0 ? 1u : 0u);
                c[2 * k + 1] = c1 + (up1 ? 1u : 0u);
                if (RECIPE == Q4_RECIPE_ZE_EDEN) {
                    // scalar sums: the terms are paired products
                    const float2 yh = make_float2(lds_f32(vl_base + c[2 * k] * 4u), lds_f32(vl_base + c[2 * k + 1] * 4u));
                    const float2 a2 = mul2_rn(y, y), b2 = mul2_rn(y, yh);
                    const int h = k >> 1;
                    pa[h] = (k & 1) ? __fadd_rn(__fadd_rn(pa[h], a2.x), a2.y) : __fadd_rn(a2.x, a2.y);
                    pb[h] = (k & 1) ? __fadd_rn(__fadd_rn(pb[h], b2.x), b2.y) : __fadd_rn(b2.x, b2.y);
                }
            }
            if (RECIPE == Q4_RECIPE_ZE_EDEN) {
                // then the lane's two groups, then the butterfly over the lanes
                float A = __fadd_rn(pa[0], pa[1]);
                float B = __fadd_rn(pb[0], pb[1]);
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    A = __fadd_rn(A, __shfl_xor_sync(0xffffffffu, A, o));
                    B = __fadd_rn(B, __shfl_xor_sync(0xffffffffu, B, o));
                }
                // A and B lie in about [1, 128] here (the block's largest element
                // has y = 1 within an ulp and code 15, level 1), inside the range
                // where the reciprocal-based quotient is exact: no division call
                sv_store = (B == 0.f) ? 0.f : __fmul_rn(s_v, div_rn_by_rcp(A, B, rcp_rn_normal<1>(B)));
            }
        }
        cv = pack8(c);
    }

    // ---- codes and scales out --------------------------------------------
    reinterpret_cast<uint32_t*>(d.mc + blk * 64)[j] = cm;
    if (!fact) reinterpret_cast<uint32_t*>(d.vc + blk * 64)[j] = cv;
    if (j == 0) {
        d.ms[blk] = s_m;
        if (!fact) d.vs[blk] = sv_store;
    }
}

// ----------------------------------------------------------------- the kernel
// URTN: the Update-RTN rounding variant of ZIP-SR; MSR: some tensor rounds
// its first moment stochastically (the LM head during its SR phase), which the
// fast path then handles too.  Separate instantiations, so that the main
// kernels carry none of that code.
// NEXTR (the next-step ZIP-SR variant) runs every tile on the general path.
template <int RECIPE, bool URTN, bool MSR, bool NEXTR>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ unsigned char smem_raw[];
    // the tables need 256-byte alignment; the launch adds 256 bytes of slack
    SmemAll& sm = *reinterpret_cast<SmemAll*>(smem_raw + ((256u - (smem_addr(smem_raw) & 255u)) & 255u));
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    WarpSmem& ws = sm.w[warp];

    if (threadIdx.x < 16) {
        const int c = threadIdx.x, c1 = c < 15 ? c + 1 : 15;
        sm.vl[c] = P.tab.vl[c];
        sm.v_rtn[c] = make_float4(P.tab.vt[c], P.tab.vl[c], P.tab.vl[c1], 0.f);
        sm.v_thr[c] = P.tab.vt[c];
        sm.v_next[c] = P.tab.vl[c1];
    }
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
        sm.lut_nf4_t[i] = P.tab.lut_nf4_t[i];
        sm.lut_nf4_l[i] = P.tab.lut_nf4_l[i];
        sm.nf4_bucket[i] = P.tab.nf4_bucket[i];
        sm.nf4_thr[i] = P.tab.nf4_bucket[i].x;
    }
    for (int i = threadIdx.x; i < kVLut / 4; i += blockDim.x) {
        reinterpret_cast<uint32_t*>(sm.lut_v_l)[i] = reinterpret_cast<const uint32_t*>(P.tab.lut_v_l)[i];
        reinterpret_cast<uint32_t*>(sm.lut_v_t)[i] = reinterpret_cast<const uint32_t*>(P.tab.lut_v_t)[i];
        if (RECIPE == Q4_RECIPE_TORCHAO)
            reinterpret_cast<uint32_t*>(sm.lut_m_log)[i] = reinterpret_cast<const uint32_t*>(P.tab.lut_m_log)[i];
    }
    if (lane == 0) {
        // count 5 per tile of a stage: the arrive (with expect_tx) of its
        // group's lead lane and the arrives that cp.async.mbarrier.arrive.noinc
        // of the group's four scale lanes trigger once their copies have landed
        for (int s = 0; s < kStageBufs; ++s) mbar_init(&ws.bar[s], 5 * kTilesPerStage);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int j = lane & 15;
    const float my_nf4 = P.tab.nf4[j], my_nf4t = P.tab.nf4_t[j];
    const float my_vl = P.tab.vl[j], my_vt = P.tab.vt[j];
    const float my_vl1 = P.tab.vl[j < 15 ? j + 1 : 15];
    // TorchAO: lane j holds the SDyn4 magnitude A_j = T_{7+j} (+inf for j >= 8)
    const float my_mag = RECIPE == Q4_RECIPE_TORCHAO ? P.tab.nf4_t[j < 8 ? 7 + j : 15] : 0.f;
    const float clip = clip_factor(P.sqnorm, P.max_norm);
    const uint64_t policy = evict_first_policy();

    // Work split: warp gw of W takes the contiguous tiles [T gw / W, T (gw+1) / W)
    // of the global tile list (within a tensor every copy source advances by a
    // constant).  A launch holds tiles of one instantiation's cost, so the
    // ranges need no finer interleaving.  Its tiles are staged kTilesPerStage
    // at a time: stage iteration i fills buffer i % kStageBufs with tiles
    // kTilesPerStage i + g of the warp's range; while the warp computes one
    // stage the next kStageBufs - 1 are in flight.
    const int64_t gw = (int64_t)blockIdx.x * kStepWarps + warp;
    const int64_t W = (int64_t)gridDim.x * kStepWarps;
    const int64_t total = P.total_pairs;
    const int64_t t_begin = total * gw / W, t_end = total * (gw + 1) / W;
    const int n_tiles = (int)(t_end - t_begin);
    if (n_tiles <= 0) return;
    const int n_st = (n_tiles + kTilesPerStage - 1) / kTilesPerStage;   // stage iterations

    // Issue cursors.  Lanes 8g..8g+7 stage tile g of every stage (g <
    // kTilesPerStage); within a group lane 0 copies the gradient, 1 the master
    // weight, 2 the m codes, 3 the v codes (bulk copies), 4, 5 the m scales and
    // 6, 7 the v scales of the tile's two blocks (4-byte copies).  Each group
    // walks its own tiles (every kTilesPerStage-th tile of the range); the
    // remaining lanes issue nothing.
    const int sl = lane & 7;
    const bool copier = lane < 8 * kTilesPerStage;
    const int grp = copier ? lane >> 3 : 0;
    const uint32_t cp_field = sl == 0 ? (uint32_t)offsetof(DevTensor, grad)
                              : sl == 1 ? (uint32_t)offsetof(DevTensor, param)
                              : sl == 2 ? (uint32_t)offsetof(DevTensor, mc)
                              : sl == 3 ? (uint32_t)offsetof(DevTensor, vc)
                              : sl < 6  ? (uint32_t)offsetof(DevTensor, ms)
                                        : (uint32_t)offsetof(DevTensor, vs);
    const uint32_t cp_dst = (uint32_t)grp * (uint32_t)sizeof(Stage) +
                            (sl == 0 ? (uint32_t)offsetof(Stage, grad)
                             : sl == 1 ? (uint32_t)offsetof(Stage, param)
                             : sl == 2 ? (uint32_t)offsetof(Stage, mc)
                             : sl == 3 ? (uint32_t)offsetof(Stage, vc)
                             : sl < 6  ? (uint32_t)offsetof(Stage, ms) + 4u * (sl & 1)
                                       : (uint32_t)offsetof(Stage, vs) + 4u * (sl & 1));
    // bytes of this lane's copy for a complete tile, and the source advance per tile
    const uint32_t cp_full = sl == 0 ? 512u : sl == 1 ? 1024u : sl < 4 ? 128u : 4u;
    const int64_t cp_step = sl == 0 ? 512 : sl == 1 ? 1024 : sl < 4 ? 128 : 8;
    const uint32_t cp_first = (sl >= 4 && (sl & 1)) ? 4u : 0u;    // second block's scale
    const uint32_t is_bulk = (copier && sl < 4) ? 1u : 0u;
    const uint32_t is_scale = (copier && sl >= 4) ? 1u : 0u;
    const uint32_t is_lead = (copier && sl == 0) ? 1u : 0u;
    const uint32_t stage0 = smem_addr(&ws.st[0][0]);
    const uint32_t bar0 = smem_addr(&ws.bar[0]);

    // this lane's group: tiles t_begin + grp, t_begin + grp + kTilesPerStage, ...
    int i_t = 0;
    {
        const int64_t t0i = t_begin + grp < t_end ? t_begin + grp : t_begin;
        int lo = 0, hi = P.n_tensors - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(P.pair_prefix + mid) <= t0i) lo = mid; else hi = mid - 1;
        }
        i_t = lo;
    }
    int64_t i_p = t_begin + grp - __ldg(P.pair_prefix + i_t);   // tile index within the tensor
    int64_t i_n = __ldg(P.pair_prefix + i_t + 1) - __ldg(P.pair_prefix + i_t);
    int64_t i_numel = 0;
    uint32_t i_bytes = 0, i_total = 0;
    bool i_fact = false;
    const char* i_src = nullptr;
    auto load_issue_tensor = [&]() {
        const DevTensor* dt = P.tensors + i_t;
        i_numel = dt->numel;
        i_fact = is_factored_recipe(RECIPE) && (RECIPE == kRecipeFactoredOnly || (dt->flags & DF_FACTORED));
        const char* base = *reinterpret_cast<const char* const*>(reinterpret_cast<const char*>(dt) + cp_field);
        i_src = base + cp_first + i_p * cp_step;
        i_bytes = (i_fact && (sl == 3 || sl >= 6)) ? 0u : cp_full;
        i_total = 1536u + 128u + (i_fact ? 0u : 128u);
    };
    load_issue_tensor();

    // Stage iteration k: the group's tile t_begin + kTilesPerStage k + grp
    // (absent past the range end); afterwards the cursor moves kTilesPerStage
    // tiles on.
    auto issue = [&](int k) {
        const int s = k % kStageBufs;
        const uint32_t bar = bar0 + 8u * (uint32_t)s;
        const uint32_t dst = stage0 + (uint32_t)s * (uint32_t)(kTilesPerStage * sizeof(Stage)) + cp_dst;
        const bool present = kTilesPerStage * k + grp < n_tiles;
        uint32_t bytes = i_bytes, total_b = i_total, staged = present ? 1u : 0u;
        if (present && i_p == i_n - 1) {
            // a tensor's last tile may hold one block and a partial block
            const int64_t left = i_numel - i_p * 2 * kBlock;
            const uint32_t nel = left >= 2 * kBlock ? 2u * kBlock : (uint32_t)left;
            const uint32_t nb = nel > (uint32_t)kBlock ? 2u : 1u;
            staged = (nel & 7u) == 0 ? 1u : 0u;
            const uint32_t b = sl & 1;
            bytes = sl < 2   ? nel * (sl == 0 ? 2u : 4u)
                    : sl < 4 ? ((sl == 3 && i_fact) ? 0u : nb * 64u)
                             : ((b < nb && (sl < 6 || !i_fact)) ? 4u : 0u);
            total_b = nel * 6u + nb * 64u * (i_fact ? 1u : 2u);
        }
        // each group's lead lane announces its tile's bulk bytes (or arrives
        // plainly for a ragged or absent tile) before any copy starts
        mbar_arrive_expect_tx_if(is_lead & staged, bar, total_b);
        mbar_arrive_if(is_lead & (staged ^ 1u), bar);
        __syncwarp();
        // the warp's earlier reads of this buffer precede the copies into it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bulk_load_if(staged & is_bulk & (bytes != 0u), dst, i_src, bytes, bar, policy);
        cp_async4_if(staged & is_scale & (bytes != 0u), dst, i_src);
        cp_async_arrive_noinc_if(is_scale, bar);
        if (present) {
            i_p += kTilesPerStage;
            i_src += kTilesPerStage * cp_step;
            if (i_p >= i_n) {
                do {
                    i_p -= i_n;
                    if (i_t + 1 >= P.n_tensors) break;
                    ++i_t;
                    i_n = __ldg(P.pair_prefix + i_t + 1) - __ldg(P.pair_prefix + i_t);
                } while (i_p >= i_n);
                load_issue_tensor();
            }
        }
    };

    for (int k = 0; k < kStageBufs - 1 && k < n_st; ++k) issue(k);
    __syncwarp();

    // Compute cursor: tile c_p of tensor c_t (one tile at a time).
    int c_t = i_t;
    {
        int lo = 0, hi = P.n_tensors - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(P.pair_prefix + mid) <= t_begin) lo = mid; else hi = mid - 1;
        }
        c_t = lo;
    }
    int64_t c_p = t_begin - __ldg(P.pair_prefix + c_t);
    int64_t c_n = __ldg(P.pair_prefix + c_t + 1) - __ldg(P.pair_prefix + c_t);
    reinterpret_cast<uint32_t*>(&ws.desc)[lane] = __ldg(reinterpret_cast<const uint32_t*>(P.tensors + c_t) + lane);
    __syncwarp();
    // factored recipe: (row, column) of the current tile's first element in
    // the parameter's matrix (a shard starts at fbase), for tensors with
    // DF_CVEC; set by one division per tensor, then advanced by 256 columns a
    // tile (at most one wrap, as cols >= 256)
    uint32_t f_row = 0, f_col = 0;
    auto fpos = [&]() {
        if (is_factored_recipe(RECIPE) && (ws.desc.flags & DF_CVEC)) {
            const int64_t e = ws.desc.fbase + c_p * 2 * kBlock;
            const int64_t r = e / ws.desc.cols;
            f_row = (uint32_t)r;
            f_col = (uint32_t)(e - r * ws.desc.cols);
            if (lane < 4) reinterpret_cast<float*>(&ws.rbv)[lane] = __ldg(ws.desc.rbar + lane);
        }
    };
    fpos();
    for (int it = 0; it < n_st; ++it) {
        if (it + kStageBufs - 1 < n_st) issue(it + kStageBufs - 1);
        const int s = it % kStageBufs;
        const bool ok = __all_sync(
            0xffffffffu, mbar_wait_bounded(&ws.bar[s], (uint32_t)((it / kStageBufs) & 1), P.wait_cycles));
        if (!ok) {
            if (lane == 0) atomicOr(P.status, ST_STAGE_TIMEOUT);
            // drain the copies this warp still has in flight (the late stage
            // included), each with the default bound, then leave
            const int last = it + kStageBufs - 1 < n_st ? it + kStageBufs - 1 : n_st - 1;
            for (int k = it; k <= last; ++k)
                (void)mbar_wait_bounded(&ws.bar[k % kStageBufs], (uint32_t)((k / kStageBufs) & 1),
                                        kDefaultWaitCycles);
            return;
        }
#pragma unroll 1
        for (int sub = 0; sub < kTilesPerStage; ++sub) {
            if (kTilesPerStage * it + sub >= n_tiles) break;
            if (c_p == c_n) {
                do {
                    ++c_t;
                } while (__ldg(P.pair_prefix + c_t + 1) == __ldg(P.pair_prefix + c_t));
                c_p = 0;
                c_n = __ldg(P.pair_prefix + c_t + 1) - __ldg(P.pair_prefix + c_t);
                reinterpret_cast<uint32_t*>(&ws.desc)[lane] =
                    __ldg(reinterpret_cast<const uint32_t*>(P.tensors + c_t) + lane);
                __syncwarp();
                fpos();
            }
            Stage& stg = ws.st[s][sub];
            const bool full = c_p < c_n - 1 || ws.desc.numel - c_p * 2 * kBlock >= 2 * kBlock;
            if (full) {
                compute_tile_full<RECIPE, URTN, MSR, NEXTR>(P, ws.desc, c_p, stg, lane, sm, ws.wt, my_nf4, my_nf4t,
                                                     my_vl, my_vt, my_vl1, my_mag, clip, f_row, f_col, ws.rbv);
            } else {
                const int64_t left = ws.desc.numel - c_p * 2 * kBlock;
                compute_tile<RECIPE, URTN, NEXTR>(P, ws.desc, c_p, (full || (left & 7) == 0) ? &stg : nullptr,
                                                  lane, sm, ws.wt, my_nf4, my_nf4t, my_vl, my_vt, clip);
            }
            ++c_p;
            if (is_factored_recipe(RECIPE)) {
                f_col += 2 * kBlock;
                if (f_col >= (uint32_t)ws.desc.cols) { f_col -= (uint32_t)ws.desc.cols; ++f_row; }
            }
            __syncwarp();
        }
    }
}

size_t step_smem_bytes() { return sizeof(SmemAll) + 256; }

template <int RECIPE, bool URTN, bool MSR, bool NEXTR>
int configure(int device) {
    static bool done[64] = {false};
    if (device < 0 || device >= 64) device = 0;
    if (done[device]) return 0;
    const cudaError_t e = cudaFuncSetAttribute(step_kernel<RECIPE, URTN, MSR, NEXTR>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)step_smem_bytes());
    if (e == cudaSuccess) done[device] = true;
    return (int)e;
}

}  // namespace

int step_grid_size(int device, int64_t total_pairs) {
    static int cached_sms[64] = {0};
    if (device < 0 || device >= 64) device = 0;
    if (cached_sms[device] == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        cached_sms[device] = sms > 0 ? sms : 1;
    }
    const int64_t full = cached_sms[device];   // one CTA per SM (shared memory holds one)
    const int64_t need = (total_pairs + kStepWarps - 1) / kStepWarps;
    return (int)(need < full ? (need > 0 ? need : 1) : full);
}

int launch_step(const StepParams& p, int grid, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    const size_t smem = step_smem_bytes();
    int ce = 0;
#define Q4_LAUNCH(R, U, M, N)                                                   \
    do {                                                                        \
        if ((ce = configure<R, U, M, N>(dev))) return ce;                       \
        step_kernel<R, U, M, N><<<grid, kStepThreads, smem, s>>>(p);            \
    } while (0)
    switch (p.recipe) {
        case Q4_RECIPE_ZIP_SR:
            if (p.v_next_r && p.v_update_rtn) Q4_LAUNCH(Q4_RECIPE_ZIP_SR, true, false, true);
            else if (p.v_next_r) Q4_LAUNCH(Q4_RECIPE_ZIP_SR, false, false, true);
            else if (p.v_update_rtn) Q4_LAUNCH(Q4_RECIPE_ZIP_SR, true, false, false);
            else if (p.has_m_sr) Q4_LAUNCH(Q4_RECIPE_ZIP_SR, false, true, false);
            else Q4_LAUNCH(Q4_RECIPE_ZIP_SR, false, false, false);
            break;
        case Q4_RECIPE_ZE_EDEN:
            if (p.has_m_sr) Q4_LAUNCH(Q4_RECIPE_ZE_EDEN, false, true, false);
            else Q4_LAUNCH(Q4_RECIPE_ZE_EDEN, false, false, false);
            break;
        case Q4_RECIPE_TORCHAO: Q4_LAUNCH(Q4_RECIPE_TORCHAO, false, false, false); break;
        case kRecipeFactoredOnly: Q4_LAUNCH(kRecipeFactoredOnly, false, false, false); break;
        default: Q4_LAUNCH(Q4_RECIPE_FACTORED, false, false, false); break;
    }
#undef Q4_LAUNCH
    return (int)cudaGetLastError();
}

}  // namespace q4
