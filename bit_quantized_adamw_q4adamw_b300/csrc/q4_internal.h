// Internal definitions of the q4adamw CUDA library (not part of the ABI).
#pragma once

#include <vector_types.h>

#include <cstddef>
#include <cstdint>

#include "q4adamw.h"

namespace q4 {

constexpr int kBlock = 128;        // elements per quantisation block
constexpr int kStepWarps = 16;     // warps per CTA of the step kernel
constexpr int kStepThreads = kStepWarps * 32;
constexpr int kVLut = 4096;        // entries of the log-bucket candidate tables
                                   // (one per bits(x)>>19 of a non-negative float)

// Per-tensor descriptor as the kernels read it (one 128-byte record).
struct DevTensor {
    float* param;
    const uint16_t* grad;
    uint16_t* bf16;
    uint8_t* mc;
    float* ms;
    uint8_t* vc;
    union {
        float* vs;         // packed v: block scales
        int64_t fbase;     // factored: matrix index of element 0 (a data-parallel
                           // shard's elem_offset; 0 for a whole tensor)
    };
    float* vrow;
    float* vcol;
    int64_t numel;
    int64_t rows;          // factored: rows of the whole parameter's matrix
    int64_t cols;          // factored: its columns (numel / rows for a whole tensor)
    uint64_t elem_offset;
    uint32_t tensor_id;
    uint32_t flags;        // DF_* bits
    float* rbar;           // factored: {mean(R), RN(1/mean(R)), 1 when every quotient
                           // R_i C_j / mean(R) is in the fast quotient's exact range, 0}
    float* colpart;        // factored: column partial sums [n_slabs][cols], then
                           // row partial sums [cov_rows][n_segs] (the rows the
                           // tensor's elements touch, 256-row slabs from the first)
};
static_assert(sizeof(DevTensor) == 128, "descriptor must stay 128 bytes");

enum : uint32_t {
    DF_M_SR = 1u,        // NF4 stochastic rounding of m this step
    DF_FACTORED = 2u,    // factored v (row/column statistics)
    DF_BF16 = 4u,        // write the BF16 weight copy
    DF_CVEC = 8u,        // factored with cols % 8 == 0, cols >= 256, rows < 2^32, 16-B aligned v_col
};

// Bits of the step's device status word (first word of the workspace).
enum : uint32_t { ST_STAGE_TIMEOUT = 1u };

// Default limit of the step kernel's wait for a staged tile: about one second
// at the SM clock.  The drain after a timed-out wait always uses it.
constexpr long long kDefaultWaitCycles = 2000000000ll;

// Codebooks and candidate tables (built on the host by q4_tables.cpp).
struct Tables {
    float nf4[16];      // m levels, ascending (NF4; SDyn4 for the TorchAO recipe)
    float nf4_t[16];    // m RTN thresholds (index 15 unused)
    float vl[16];       // v levels for this launch (Dyn4 or Dyn4-NZ)
    float vt[16];       // v RTN thresholds (index 15 unused)
    uint8_t lut_nf4_t[64];   // NF4 threshold candidate by linear bucket
    uint8_t lut_nf4_l[64];   // NF4 level (cell) candidate by linear bucket
    uint8_t lut_v_l[kVLut];  // v level (cell) candidate by log bucket
    uint8_t lut_v_t[kVLut];  // v threshold candidate by log bucket
    float2 nf4_bucket[64];   // NF4 RTN by linear bucket: {threshold of the candidate, candidate}
    uint8_t lut_m_log[kVLut];  // SDyn4 RTN: lower bound of #{i : A_i <= |m|/s} by log bucket
    int m_lut;               // 1 when the linear-bucket tables are valid for the m codebook
};

// Host-side tables: 0 = NF4, 1 = Dyn4, 2 = Dyn4-NZ, 3 = SDyn4, 4 = Lin4-NZ.
struct Codebook {
    float levels[16];
    float thresholds[15];
};
const Codebook& codebook(int which);
// Fills t for the m codebook `mbook` (0 or 3) and the v codebook `vbook`
// (1, 2 or 4).  Returns false if a v candidate table cannot be built (never
// for the shipped codebooks).
bool build_tables(int mbook, int vbook, Tables* t);

struct StepParams {
    const DevTensor* tensors;
    uint32_t* status;             // device status word, zeroed by the upload
    const int64_t* pair_prefix;   // n+1 entries: first block-pair of each tensor
    int64_t total_pairs;
    int n_tensors;
    int recipe;
    float beta1, beta2, omb1, omb2, c2, eps, decay, step_size;
    uint32_t step;
    int fast_math;                // eps and c2 keep 1/(sqrt(v) c2 + eps) in the fast domain
    int v_update_rtn;             // ZIP-SR with Update-RTN in place of Update-SR
    int v_next_r;                 // ZIP-SR rounds in the next step's zero-gradient preconditioner
    float c2_next;                //   its 1/sqrt(1 - beta2^(t+1))
    int has_m_sr;                 // some tensor rounds its first moment stochastically
    const float* sqnorm;          // global-norm clipping: device sum of squares, or NULL
    float max_norm;               //   and the clipping threshold
    long long wait_cycles;        // limit of a warp's wait for a staged tile (SM clock cycles)
    // the step scalars broadcast to pairs, for the paired FP32 instructions
    float2 x2_beta1, x2_beta2, x2_omb1, x2_omb2, x2_c2, x2_eps, x2_decay, x2_neg_step;
    uint32_t round_keys[20];      // Philox key schedule: (k0, k1) for rounds 0..9
    Tables tab;
};

struct FactoredParams {
    const DevTensor* tensors;
    const int64_t* row_prefix;    // n+1: factored rows of each tensor (its whole matrix)
    const int64_t* tile_prefix;   // n+1: column tiles (slab x segment) of each tensor
    const int64_t* col_prefix;    // n+1: factored columns of each tensor
    const int32_t* factored_ids;  // tensor index of the k-th factored tensor
    int n_tensors;
    int n_factored;
    int64_t total_rows, total_tiles, total_cols;
    float beta2, omb2;
    const float* sqnorm;          // as StepParams
    float max_norm;
    float* sums;                  // data-parallel: per factored tensor, row sums [rows] then
                                  // column sums [cols], at row_prefix[t] + col_prefix[t]
};

// Rows of a factored tensor's matrix that its elements [fbase, fbase + numel)
// touch: the first, and how many.
__host__ __device__ inline void covered_rows(int64_t fbase, int64_t numel, int64_t cols, int64_t* first,
                                             int64_t* count) {
    *first = fbase / cols;
    *count = numel > 0 ? (fbase + numel - 1) / cols - *first + 1 : 0;
}

// Gradient sum of squares (global-norm clipping).  Chunks are aligned runs of
// kNormChunkTiles 256-element tiles of one tensor.
struct NormTensor {
    const uint16_t* grad;
    int64_t numel;
};
constexpr int kNormWarps = 8;
constexpr int kNormGroupsPerWarp = 8;                              // 32 tiles per group
constexpr int64_t kNormChunkTiles = kNormWarps * kNormGroupsPerWarp * 32;   // 2048
struct NormParams {
    const NormTensor* tensors;
    const int64_t* chunk_prefix;  // n+1: chunks of each tensor
    int n_tensors;
    int64_t total_chunks;
    float* partials;              // total_chunks: chunk sums, reduced in place
    float* tensor_sums;           // n
    float* out;                   // the sum of squares
};

// Count of non-finite BF16 gradients: runs of 8 elements per tensor.
struct NonfiniteParams {
    const NormTensor* tensors;
    const int64_t* run_prefix;    // n+1: runs of each tensor
    int n_tensors;
    int64_t total_runs;
    unsigned long long* out;      // the count (zeroed by the launch)
};

// Kernel-internal recipe value: the factored recipe on a launch whose tensors
// are all factored (rank >= 2), which compiles without the packed-v code.
constexpr int kRecipeFactoredOnly = 16;
__host__ __device__ constexpr bool is_factored_recipe(int recipe) {
    return recipe == Q4_RECIPE_FACTORED || recipe == kRecipeFactoredOnly;
}

constexpr int kSlabRows = 256;     // rows per column-partial slab (8 warps x 32 rows)
constexpr int kSegCols = 256;      // columns per row-partial segment (32 lanes x 8)

// Philox4x32-10 key schedule of a 64-bit seed: (k0, k1) of rounds 0..9, the
// Weyl increments 0x9E3779B9 and 0xBB67AE85 added once per round.
inline void philox_round_keys(uint64_t seed, uint32_t rk[20]) {
    const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        rk[2 * r] = k0 + (uint32_t)r * 0x9E3779B9u;
        rk[2 * r + 1] = k1 + (uint32_t)r * 0xBB67AE85u;
    }
}

// Records a cudaError_t for q4adamw_last_cuda_error() and returns Q4_ECUDA.
int record_cuda_error(int cuda_error);

// Launchers (return cudaError_t as int).
int launch_step(const StepParams& p, int grid, void* stream);
int step_grid_size(int device, int64_t total_pairs);
int launch_factored(const FactoredParams& p, void* stream);
// Data-parallel factored statistics: this shard's row/column sums into p.sums
// (statistics pass, then the sums), and the update of R and C from sums over
// all shards followed by mean(R).
int launch_factored_sums(const FactoredParams& p, void* stream);
int launch_factored_from_sums(const FactoredParams& p, void* stream);
int launch_grad_sqnorm(const NormParams& p, int device, void* stream);
int launch_nonfinite(const NonfiniteParams& p, int device, void* stream);
int launch_draws(uint64_t seed, uint32_t step, uint32_t tensor_id, uint64_t idx0, uint32_t purpose, int64_t n,
                 uint32_t* out, void* stream);
int launch_dequant(const DevTensor& d, int recipe, const float* nf4, const float* vl, float* m_out, float* v_out,
                   void* stream);

}  // namespace q4
