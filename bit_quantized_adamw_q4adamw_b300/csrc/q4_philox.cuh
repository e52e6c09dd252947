// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11) as the step kernel draws it: key = (seed low, seed
// high), counter = (idx >> 2, (idx >> 34) | purpose << 28, tensor id, step), and
// the draw of element idx is word idx & 3.  The round keys (the key schedule,
// q4::philox_round_keys) are computed on the host.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace q4 {

// Ten rounds from a precomputed key schedule; each round's two 32x32->64
// products are single wide multiplies.
__device__ __forceinline__ uint4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, const uint32_t* rk) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)c0 * 0xD2511F53u;
        const uint64_t p1 = (uint64_t)c2 * 0xCD9E8D57u;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ rk[2 * r];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ rk[2 * r + 1];
        c0 = n0;
        c1 = (uint32_t)p1;
        c2 = n2;
        c3 = (uint32_t)p0;
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

}  // namespace q4
