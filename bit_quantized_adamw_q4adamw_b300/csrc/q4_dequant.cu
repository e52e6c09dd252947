// State decoding for export, checkpoint inspection and tests:
// m = NF4[q] * s_m; v = V[q] * s_v (packed) or R_i * C_j / mean(R) (factored).
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_internal.h"
#include "q4_reduce.cuh"

namespace q4 {

namespace {

struct DequantParams {
    DevTensor d;
    float nf4[16];
    float vl[16];
    float* m_out;
    float* v_out;
    int factored;
};

__global__ void __launch_bounds__(256) dequant_kernel(const __grid_constant__ DequantParams P) {
    __shared__ float red[256];
    const DevTensor& d = P.d;
    float rbar = 0.f;
    if (P.factored && P.v_out) rbar = block_mean(d.vrow, d.rows, red);
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < d.numel; e += (int64_t)gridDim.x * 256) {
        const int64_t b = e / kBlock;
        const int sh = (int)(e & 1) * 4;
        if (P.m_out) P.m_out[e] = __fmul_rn(P.nf4[(d.mc[e >> 1] >> sh) & 15], d.ms[b]);
        if (P.v_out) {
            if (P.factored) {
                const int64_t i = e / d.cols, j = e - i * d.cols;
                P.v_out[e] = (rbar == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(d.vrow[i], d.vcol[j]), rbar);
            } else {
                P.v_out[e] = __fmul_rn(P.vl[(d.vc[e >> 1] >> sh) & 15], d.vs[b]);
            }
        }
    }
}

}  // namespace

int launch_dequant(const DevTensor& d, int recipe, const float* nf4, const float* vl, float* m_out, float* v_out,
                   void* stream) {
    DequantParams p{};
    p.d = d;
    for (int k = 0; k < 16; ++k) {
        p.nf4[k] = nf4[k];
        p.vl[k] = vl[k];
    }
    p.m_out = m_out;
    p.v_out = v_out;
    p.factored = (recipe == Q4_RECIPE_FACTORED) && (d.flags & DF_FACTORED);
    int64_t g = (d.numel + 255) / 256;
    if (g > 148 * 8) g = 148 * 8;
    if (g < 1) g = 1;
    dequant_kernel<<<(int)g, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace q4
