// Factored second-moment statistics for rank >= 2 tensors (AReno docs
// "4-bit AdamW", section "State representation": as in Adafactor, means of
// g^2 over the rows and over the columns of the [shape[0], -1] view, kept as
// exponential averages; 1-D tensors keep packed 4-bit v).
//
// Three launches, all multi-tensor and deterministic (fixed summation order,
// no atomics).  A tensor may be one data-parallel shard of its parameter (the
// same page: each rank's row and column sums of g^2 are added over the group,
// and R and C take their exponential update from the totals): its elements are [fbase, fbase + numel) of the
// whole [rows, cols] matrix, the pass covers the rows they touch, and the
// rows/cols kernels either write the shard's row and column sums for the
// caller to add over the ranks, or update R and C from the added sums.
//   stats_kernel    persistent CTAs of 8 warps, four per SM, each taking tiles
//                   of 256 rows x 256 columns of a tensor in turn: g is read
//                   once, 16 bytes (8 BF16) per lane and row.
//                   Each lane sums the 8 squares of its row chunk; each of a
//                   warp's 32 rows is summed over the lanes with the pairing of
//                   an xor butterfly (lane offsets 16, 8, 4, 2, 1), giving row
//                   partials per 256-column segment.  A strip of 32 rows that
//                   lies wholly inside the tensor's elements is read as 4
//                   batches of 8 independent loads per lane; edge strips take a
//                   per-row checked path with the same pairing (a transpose
//                   tree, lane l ending with row l's sum).  Column sums over the
//                   warp's 32 rows are combined over the 8 warps in warp order,
//                   giving column partials per 256-row slab.
//   rows_kernel,    a row's partials summed in segment order by one thread, a
//   cols_kernel     column's over its slabs by one CTA of 8 warps (contiguous
//                   slab ranges per warp, then the warps in order); mean = sum /
//                   cols (rows), and the average R_i <- beta2 R_i + (1-beta2)
//                   mean (C_j likewise).
//   rbar_kernel     one 1024-thread CTA per factored tensor: mean(R) in a fixed
//                   tree order, stored with its correctly rounded reciprocal.
// The step kernel then forms vhat_ij = R_i * C_j / mean(R) per element (with
// the global-norm clip factor, when given, applied to g before squaring here).
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_reduce.cuh"

namespace q4 {
namespace {
// x >= 0 lies in {0} or [2^-100, 2^100]: the quotient's safe range.
__device__ __forceinline__ bool quot_range_ok(float x) {
    const uint32_t b = __float_as_uint(x);
    return b == 0u || (b - 0x0d800000u) <= (0x71800000u - 0x0d800000u);
}
}  // namespace
}  // namespace q4

namespace q4 {

namespace {

constexpr int kStatsWarps = kSlabRows / 32;   // 8 warps, 32 rows each

__device__ __forceinline__ float bf16f(uint32_t h) { return __uint_as_float(h << 16); }

// Four CTAs per SM (64 registers), and a grid of exactly that many CTAs
// striding over the tiles: measured faster than three per SM or a larger grid.
constexpr int kStatsCtasPerSm = 4;

__global__ void __launch_bounds__(kStatsWarps * 32, kStatsCtasPerSm) stats_kernel(const __grid_constant__ FactoredParams P) {
    __shared__ float colsum[kStatsWarps][kSegCols];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float clip = clip_factor(P.sqnorm, P.max_norm);   // 1 without clipping
    for (int64_t tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
        const int t = find_tensor(P.tile_prefix, P.n_tensors, tile);
        const DevTensor& d = P.tensors[t];
        const int64_t local = tile - __ldg(P.tile_prefix + t);
        const int64_t cols = d.cols, fbase = d.fbase, fend = d.fbase + d.numel;
        // the rows of the matrix this tensor's elements [fbase, fend) touch
        // (all of them for a whole tensor); slabs count from the first
        int64_t r_first, cov;
        covered_rows(fbase, d.numel, cols, &r_first, &cov);
        const int64_t nseg = (cols + kSegCols - 1) / kSegCols;
        const int64_t slab = local / nseg, seg = local - slab * nseg;
        const int64_t r0 = slab * kSlabRows + warp * 32;
        const int64_t c0 = seg * kSegCols + lane * 8;
        const int nc = c0 >= cols ? 0 : (cols - c0 >= 8 ? 8 : (int)(cols - c0));
        const bool vec = nc == 8 && (cols & 7) == 0;
        float col[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float my_row = 0.f;   // the sum of row r0 + lane over this segment
        // interior strip (warp-uniform): all 32 rows in range, the segment's
        // 256 columns inside the matrix, every element inside [fbase, fend)
        const bool interior = (cols & 7) == 0 && seg * kSegCols + kSegCols <= cols && r0 + 32 <= cov &&
                              (r_first + r0) * cols + seg * kSegCols >= fbase &&
                              (r_first + r0 + 31) * cols + (seg + 1) * kSegCols <= fend;
        if (interior) {
            // 4 batches of 8 independent 16-byte loads per lane; each row's sum
            // over the 32 lanes by an xor butterfly (offsets 16, 8, 4, 2, 1),
            // kept by lane (row - r0)
            const uint16_t* g0 = d.grad + ((r_first + r0) * cols + c0 - fbase);
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                uint4 w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = __ldcs(reinterpret_cast<const uint4*>(g0 + (int64_t)(8 * b + i) * cols));
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t h[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
                    float sq[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = __fmul_rn(bf16f(h[k] & 0xffffu), clip);
                        const float hi = __fmul_rn(bf16f(h[k] >> 16), clip);
                        sq[2 * k] = __fmul_rn(lo, lo);
                        sq[2 * k + 1] = __fmul_rn(hi, hi);
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) col[k] = __fadd_rn(col[k], sq[k]);
                    float rs = __fadd_rn(__fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3])),
                                         __fadd_rn(__fadd_rn(sq[4], sq[5]), __fadd_rn(sq[6], sq[7])));
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, o));
                    if (lane == 8 * b + i) my_row = rs;
                }
            }
        } else {
            float rowp[32];
    #pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int64_t r = r0 + i;
                float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (r < cov && nc > 0) {
                    const int64_t ge = (r_first + r) * cols + c0;   // matrix index of the lane's first column
                    const uint16_t* g = d.grad + (ge - fbase);
                    if (vec) {
                        // fbase and cols are multiples of 8: a run of 8 lies wholly inside or outside
                        if (ge >= fbase && ge < fend) {
                            const uint4 w = __ldcs(reinterpret_cast<const uint4*>(g));
                            const uint32_t h[4] = {w.x, w.y, w.z, w.w};
    #pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float lo = __fmul_rn(bf16f(h[k] & 0xffffu), clip);
                                const float hi = __fmul_rn(bf16f(h[k] >> 16), clip);
                                sq[2 * k] = __fmul_rn(lo, lo);
                                sq[2 * k + 1] = __fmul_rn(hi, hi);
                            }
                        }
                    } else {
    #pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (k < nc && ge + k >= fbase && ge + k < fend) {
                                const float x = __fmul_rn(bf16f(g[k]), clip);
                                sq[k] = __fmul_rn(x, x);
                            }
                        }
                    }
                }
    #pragma unroll
                for (int k = 0; k < 8; ++k) col[k] = __fadd_rn(col[k], sq[k]);
                rowp[i] = __fadd_rn(__fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3])),
                                    __fadd_rn(__fadd_rn(sq[4], sq[5]), __fadd_rn(sq[6], sq[7])));
            }
            // transpose reduction: afterwards rowp[0] of lane l is the sum over the
            // 32 lanes of row l (a fixed tree)
    #pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool upper = (lane & o) != 0;
    #pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = upper ? rowp[i] : rowp[i + o];
                    const float keep = upper ? rowp[i + o] : rowp[i];
                    rowp[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
                }
            }
            my_row = rowp[0];
        }
        const int64_t nslab = (cov + kSlabRows - 1) / kSlabRows;
        if (r0 + lane < cov) d.colpart[nslab * cols + (r0 + lane) * nseg + seg] = my_row;
#pragma unroll
        for (int k = 0; k < 8; ++k) colsum[warp][lane * 8 + k] = col[k];
        __syncthreads();
        {
            const int c = threadIdx.x;                 // column within the segment
            float s = colsum[0][c];
#pragma unroll
            for (int w = 1; w < kStatsWarps; ++w) s = __fadd_rn(s, colsum[w][c]);
            const int64_t col_g = seg * kSegCols + c;
            if (col_g < cols) d.colpart[slab * cols + col_g] = s;
        }
        __syncthreads();
    }
}

// Sum of a row's partials over its segments and of a column's over its
// slabs, in segment (slab) order; rows the tensor does not touch sum to 0.
__device__ __forceinline__ float row_sum(const DevTensor& d, int64_t i) {
    int64_t r_first, cov;
    covered_rows(d.fbase, d.numel, d.cols, &r_first, &cov);
    if (i < r_first || i >= r_first + cov) return 0.f;
    const int64_t nseg = (d.cols + kSegCols - 1) / kSegCols;
    const int64_t nslab = (cov + kSlabRows - 1) / kSlabRows;
    const float* p = d.colpart + nslab * d.cols + (i - r_first) * nseg;
    float acc = __ldg(p);
    for (int64_t q = 1; q < nseg; ++q) acc = __fadd_rn(acc, __ldg(p + q));
    return acc;
}
// Column j's sum over its slab partials by one CTA of kColWarps warps, each
// lane one column: warp w adds the slabs [w q, (w+1) q) left to right (q =
// ceil(nslab / kColWarps)), then the warp results are added in warp order.
// Empty ranges contribute +0, which leaves a sum of squares unchanged, so with
// at most kColWarps slabs this is the sequential sum.  Every thread of the
// CTA must call it (it synchronises); lanes without a column pass valid =
// false and get 0.
constexpr int kColWarps = 8;
__device__ __forceinline__ float col_sum_cta(const DevTensor& d, int64_t j, bool valid, float (*red)[32]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc = 0.f;
    if (valid) {
        int64_t r_first, cov;
        covered_rows(d.fbase, d.numel, d.cols, &r_first, &cov);
        const int64_t nslab = (cov + kSlabRows - 1) / kSlabRows;
        const int64_t q = (nslab + kColWarps - 1) / kColWarps;
        const int64_t s0 = warp * q, s1 = s0 + q < nslab ? s0 + q : nslab;
        for (int64_t s = s0; s < s1; ++s) acc = __fadd_rn(acc, __ldg(d.colpart + s * d.cols + j));
    }
    red[warp][lane] = acc;
    __syncthreads();
    float tot = red[0][lane];
#pragma unroll
    for (int w = 1; w < kColWarps; ++w) tot = __fadd_rn(tot, red[w][lane]);
    __syncthreads();
    return tot;
}

// One thread per factored row: R_i from its segment partials (finalize) or
// from the summed sums (data-parallel); or this shard's row sum into P.sums.
enum { ROWS_FINALIZE = 0, ROWS_SUMS = 1, ROWS_FROM_SUMS = 2 };
template <int MODE>
__global__ void __launch_bounds__(256) rows_kernel(const __grid_constant__ FactoredParams P) {
    for (int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x; idx < P.total_rows; idx += (int64_t)gridDim.x * 256) {
        const int t = find_tensor(P.row_prefix, P.n_tensors, idx);
        const DevTensor& d = P.tensors[t];
        const int64_t i = idx - __ldg(P.row_prefix + t);
        float* sums = P.sums + __ldg(P.row_prefix + t) + __ldg(P.col_prefix + t);
        if (MODE == ROWS_SUMS) {
            sums[i] = row_sum(d, i);
        } else {
            const float acc = MODE == ROWS_FINALIZE ? row_sum(d, i) : __ldg(sums + i);
            d.vrow[i] = __fmaf_rn(P.beta2, d.vrow[i], __fmul_rn(P.omb2, __fdiv_rn(acc, (float)d.cols)));
        }
    }
}

// Factored columns, kColWarps warps per CTA over 32 columns of the global
// column list (a tensor boundary may fall inside a CTA's columns): C_j from
// its slab partials (finalize), this shard's column sum into P.sums, or C_j
// from the summed sums (data-parallel).
template <int MODE>
__global__ void __launch_bounds__(kColWarps * 32) cols_kernel(const __grid_constant__ FactoredParams P) {
    __shared__ float red[kColWarps][32];
    const int lane = threadIdx.x & 31;
    for (int64_t base = (int64_t)blockIdx.x * 32; base < P.total_cols; base += (int64_t)gridDim.x * 32) {
        const int64_t g = base + lane;
        const bool valid = g < P.total_cols;
        const int64_t gc = valid ? g : P.total_cols - 1;
        const int t = find_tensor(P.col_prefix, P.n_tensors, gc);
        const DevTensor& d = P.tensors[t];
        const int64_t j = gc - __ldg(P.col_prefix + t);
        float* sums = P.sums + __ldg(P.row_prefix + t) + __ldg(P.col_prefix + t) + d.rows;
        const float acc = MODE == ROWS_FROM_SUMS ? (valid ? __ldg(sums + j) : 0.f) : col_sum_cta(d, j, valid, red);
        if (valid && (threadIdx.x >> 5) == 0) {
            if (MODE == ROWS_SUMS) sums[j] = acc;
            else d.vcol[j] = __fmaf_rn(P.beta2, d.vcol[j], __fmul_rn(P.omb2, __fdiv_rn(acc, (float)d.rows)));
        }
    }
}

// mean(R) of each factored tensor by one CTA of kRbarThreads threads (the
// fixed order of block_mean), with its correctly rounded reciprocal, and
// whether every quotient R_i C_j / mean(R) of the tensor is in the range
// where the step's reciprocal-based quotient is exact: from the largest and
// the smallest nonzero R_i and C_j (on the bit patterns of these non-negative
// floats: NaN and +inf above every finite value), every nonzero product and
// quotient lies between the rounded products and quotients of the extremes
// (rounding is monotone), which must lie in [2^-100, 2^100] (the quotients
// with a factor-2 margin).  Stored as {mean, 1/mean, 1 or 0, 0}.
constexpr int kRbarThreads = 1024;
__device__ __forceinline__ void minmax_bits(const float* x, int64_t n, uint32_t& mx, uint32_t& mn_m1, uint32_t* red) {
    uint32_t a = 0u, b = 0xffffffffu;
    for (int64_t i = threadIdx.x; i < n; i += kRbarThreads) {
        const uint32_t u = __float_as_uint(x[i]);
        a = max(a, u);
        b = min(b, u - 1u);   // the smallest nonzero, minus 1 (all ones: none)
    }
    a = __reduce_max_sync(0xffffffffu, a);
    b = __reduce_min_sync(0xffffffffu, b);
    if ((threadIdx.x & 31) == 0) { red[2 * (threadIdx.x >> 5)] = a; red[2 * (threadIdx.x >> 5) + 1] = b; }
    __syncthreads();
    if (threadIdx.x < 32) {
        a = red[2 * threadIdx.x];
        b = red[2 * threadIdx.x + 1];
        a = __reduce_max_sync(0xffffffffu, a);
        b = __reduce_min_sync(0xffffffffu, b);
    }
    mx = a;
    mn_m1 = b;
    __syncthreads();
}
__global__ void __launch_bounds__(kRbarThreads) rbar_kernel(const __grid_constant__ FactoredParams P) {
    __shared__ float red[kRbarThreads];
    __shared__ uint32_t redu[64];
    for (int k = blockIdx.x; k < P.n_factored; k += gridDim.x) {
        const DevTensor& d = P.tensors[__ldg(P.factored_ids + k)];
        const float mean = block_mean<kRbarThreads>(d.vrow, d.rows, red);
        uint32_t rmax, rmin_m1, cmax, cmin_m1;
        minmax_bits(d.vrow, d.rows, rmax, rmin_m1, redu);
        minmax_bits(d.vcol, d.cols, cmax, cmin_m1, redu);
        if (threadIdx.x == 0) {
            const float y = __frcp_rn(mean);
            const bool rb_ok = mean != 0.f && quot_range_ok(mean);
            bool fast = rb_ok;
            if (rb_ok && rmin_m1 != 0xffffffffu && cmin_m1 != 0xffffffffu) {
                const float pmax = __fmul_rn(__uint_as_float(rmax), __uint_as_float(cmax));
                const float pmin = __fmul_rn(__uint_as_float(rmin_m1 + 1u), __uint_as_float(cmin_m1 + 1u));
                fast = quot_range_ok(pmax) && quot_range_ok(pmin) && pmin != 0.f &&
                       __fdiv_rn(pmin, mean) >= 0x1p-99f && __fdiv_rn(pmax, mean) <= 0x1p99f;
            }
            *reinterpret_cast<float4*>(d.rbar) = make_float4(mean, y, fast ? 1.f : 0.f, 0.f);
        }
    }
}

int grid_for(int64_t work, int per_cta, int64_t cap) {
    int64_t g = (work + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

int sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 148;
    return sms;
}

void launch_stats(const FactoredParams& p, cudaStream_t s) {
    if (p.total_tiles > 0)
        stats_kernel<<<grid_for(p.total_tiles, 1, (int64_t)sm_count() * kStatsCtasPerSm), kStatsWarps * 32, 0, s>>>(
            p);
}

template <int MODE>
void launch_rows_cols(const FactoredParams& p, cudaStream_t s) {
    if (p.total_rows > 0) rows_kernel<MODE><<<grid_for(p.total_rows, 256, 148 * 16), 256, 0, s>>>(p);
    if (p.total_cols > 0) cols_kernel<MODE><<<grid_for(p.total_cols, 32, 148 * 64), kColWarps * 32, 0, s>>>(p);
}

}  // namespace

int launch_factored(const FactoredParams& p, void* stream) {
    if (p.n_factored == 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_stats(p, s);
    launch_rows_cols<ROWS_FINALIZE>(p, s);
    rbar_kernel<<<p.n_factored < 1024 ? p.n_factored : 1024, kRbarThreads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

int launch_factored_sums(const FactoredParams& p, void* stream) {
    if (p.n_factored == 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_stats(p, s);
    launch_rows_cols<ROWS_SUMS>(p, s);
    return (int)cudaGetLastError();
}

int launch_factored_from_sums(const FactoredParams& p, void* stream) {
    if (p.n_factored == 0) return 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    launch_rows_cols<ROWS_FROM_SUMS>(p, s);
    rbar_kernel<<<p.n_factored < 1024 ? p.n_factored : 1024, kRbarThreads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
