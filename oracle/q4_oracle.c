/*
 * q4_oracle.c -- CPU oracle for the fused 4-bit AdamW step (ZIP-SR / ZE-EDEN).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py may load this library.  The product path
 * (the CUDA library under bit_quantized_adamw_q4adamw_b300/csrc) never
 * calls it and shares no code, header, table or generator with it.
 *
 * Plain, slow, single-threaded.  Build with -O2 -ffp-contract=off and no
 * fast-math: every FP32 operation below is one correctly rounded IEEE
 * operation, written out in the order the method states it; a fused
 * multiply-add appears only where fmaf() is written.
 *
 * Sources (cited by page title and section):
 *  - "Rounding in Preconditioner Space: Redesigning 4-bit AdamW
 *    Optimizer-State Quantization" (Li et al., arXiv:2610.12444), listing
 *    page: Abstract (moment recurrences, ZIP-SR, ZE-EDEN, NF4 first moment,
 *    LM-head SR in the final 10%), Table 1 (State-RTN / State-SR /
 *    Update-RTN / Update-SR near-zero cell), Table 2 (recipe per buffer).
 *  - "Two 4-bit AdamW methods brought..." news page, paragraphs 2-4 (FP32
 *    master weights, the two running buffers, preconditioner-space rounding,
 *    packed values plus block scales = 1.0625 bytes/param).
 *  - AReno docs "4-bit AdamW", section "State representation" (parameter-
 *    local 128-element blocks, zero-excluding map for 1-D v, Adafactor row /
 *    column means over [shape[0], -1]) and "Requirements and errors" (one
 *    fused kernel whose FP32 work per block is local and of fixed size).
 * Where those pages are silent, the reading taken is stated at the function.
 *
 * Parity status of each function is given in oracle/oracle.py's header.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OB 128 /* block size: AReno docs "4-bit AdamW", State representation */

enum { OR_ZIP_SR = 0, OR_ZE_EDEN = 1, OR_FACTORED = 2, OR_TORCHAO = 3 };
enum { OT_LM_HEAD = 1u, OT_FACTORED = 2u };
/* Per-call flags: the LM-head SR phase (Table 2 note) and two rounding
 * variants of the listing page's ablations: State-SR for the first moment of
 * every tensor, and Update-RTN in place of Update-SR under ZIP-SR (Table 1
 * rules). */
enum { OS_LM_HEAD_SR_ACTIVE = 1u, OS_M_SR_ALL = 2u, OS_V_UPDATE_RTN = 4u, OS_V_NEXT_R = 8u };
enum { OP_M_SR = 0u, OP_V_SR = 1u };

/* ------------------------------------------------------------------ */
/* BF16 <-> FP32 (bit-level definitions of the format)                  */
/* ------------------------------------------------------------------ */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even FP32 -> BF16 (finite inputs). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers:  */
/* as easy as 1, 2, 3", SC'11).  The pages name no generator; a counter- */
/* based one keyed by (seed, step, tensor id, element) is the reading.   */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u; /* Weyl key bumps */
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit draw for element `idx` (global index within its parameter)
 * of stream `purpose`: counter = (idx>>2, (idx>>34) | purpose<<28,
 * tensor_id, step), key = (seed_lo, seed_hi); word idx&3 is used. */
uint32_t oracle_draw(uint64_t seed, uint32_t step, uint32_t tensor_id, uint64_t idx, uint32_t purpose) {
    uint32_t ctr[4] = {(uint32_t)(idx >> 2), (uint32_t)(idx >> 34) | (purpose << 28), tensor_id, step};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[idx & 3u];
}

/* Uniform in [0,1) with 24 random bits: u = (w >> 8) * 2^-24 (exact). */
float oracle_uniform(uint32_t w) { return (float)(w >> 8) * 0x1p-24f; }

/* ------------------------------------------------------------------ */
/* Host scalars: computed in double, each rounded once to FP32.          */
/* out = {bc1, c2, step_size, decay, omb1, omb2}.                        */
/* AdamW as in torch.optim.AdamW (decoupled weight decay, bias-corrected */
/* moments): news page paragraph 2; listing page Abstract.              */
/* ------------------------------------------------------------------ */
void oracle_host_scalars(float lr, float beta1, float beta2, float weight_decay, int64_t t, float out[6]) {
    double dlr = lr, d1 = beta1, d2 = beta2, dwd = weight_decay;
    double bc1 = 1.0 - pow(d1, (double)t);
    double bc2 = 1.0 - pow(d2, (double)t);
    out[0] = (float)bc1;
    out[1] = (float)(1.0 / sqrt(bc2));
    out[2] = (float)(dlr / bc1);
    out[3] = (float)(1.0 - dlr * dwd);
    out[4] = (float)(1.0 - d1);
    out[5] = (float)(1.0 - d2);
}

typedef struct {
    float beta1, beta2, eps;
    float c2, step_size, decay, omb1, omb2;
    float rb, rc;   /* the rules' preconditioner space: r(x) = 1 / (sqrt(rb * x) * rc + eps) */
} scal_t;

static scal_t make_scalars(float lr, float beta1, float beta2, float eps, float wd, int64_t t) {
    float h[6];
    oracle_host_scalars(lr, beta1, beta2, wd, t, h);
    scal_t s;
    s.beta1 = beta1; s.beta2 = beta2; s.eps = eps;
    s.c2 = h[1]; s.step_size = h[2]; s.decay = h[3]; s.omb1 = h[4]; s.omb2 = h[5];
    s.rb = 1.0f; s.rc = s.c2;
    return s;
}

/* Preconditioner r(x) = 1 / (sqrt(x) * c2 + eps): the quantity in which
 * ZIP-SR chooses its rounding probabilities (listing page Abstract,
 * Table 1 "Precond. error"). */
static float precond(float x, const scal_t* s) { return 1.0f / (sqrtf(x) * s->c2 + s->eps); }

/* The preconditioner in which the Update rules round.  By default rb = 1,
 * rc = c2, so rule_r(x) = precond(x) exactly (1 * x is exact): the r the
 * update of the same step used.  The next-step variant (Table 1 evaluates
 * the preconditioner error at step t+1 with |g_{t+1}| = O(eps)) takes the
 * next step's zero-gradient preconditioner: rb = beta2, rc = 1 /
 * sqrt(1 - beta2^(t+1)). */
static float rule_r(float x, const scal_t* s) { return 1.0f / (sqrtf(s->rb * x) * s->rc + s->eps); }

/* ------------------------------------------------------------------ */
/* Rounding rules on one value, given the block's scaled levels          */
/* a_k = L_k * s (ascending) and RTN thresholds T_k = t_k * s.           */
/* Listing page Table 1 names the four rules; Table 2 assigns them.     */
/* ------------------------------------------------------------------ */

/* State-RTN: code = #{k in 0..14 : x > T_k} (nearest level; a tie at a
 * threshold goes to the lower code). */
static int rule_state_rtn(const float T[15], float x) {
    int c = 0;
    for (int k = 0; k < 15; ++k)
        if (x > T[k]) c++;
    return c;
}

/* Cell index: max{k : a_k <= x}, 0 when no level is <= x. */
static int cell_of(const float a[16], float x) {
    int k = 0;
    for (int j = 0; j < 16; ++j)
        if (a[j] <= x) k = j;
    return k;
}

/* State-SR: up with probability (x - a_k)/(a_{k+1} - a_k), decided as
 * u*(a_{k+1}-a_k) < x-a_k.  Unbiased in the state: E[Q] = x. */
static int rule_state_sr(const float a[16], float x, float u) {
    int k = cell_of(a, x);
    if (k == 15) return 15;
    return (u * (a[k + 1] - a[k]) < (x - a[k])) ? k + 1 : k;
}

/* Update-SR (ZIP-SR): up with probability (r_k - r)/(r_k - r_{k+1}) in
 * preconditioner space, so E[r(Q)] = r(x).  r is r(x) as used by the
 * update of the same step. */
static int rule_update_sr(const float a[16], float x, float r, float u, const scal_t* s) {
    int k = cell_of(a, x);
    if (k == 15) return 15;
    float rk = rule_r(a[k], s);
    float rk1 = rule_r(a[k + 1], s);
    return (u * (rk - rk1) < (rk - r)) ? k + 1 : k;
}

/* Update-RTN: the adjacent level whose preconditioner is nearer to r; a
 * tie goes to the lower code. */
static int rule_update_rtn(const float a[16], float x, float r, const scal_t* s) {
    int k = cell_of(a, x);
    if (k == 15) return 15;
    float rk = rule_r(a[k], s);
    float rk1 = rule_r(a[k + 1], s);
    return ((r - rk1) < (rk - r)) ? k + 1 : k;
}

enum { RULE_STATE_RTN = 0, RULE_STATE_SR = 1, RULE_UPDATE_RTN = 2, RULE_UPDATE_SR = 3 };

static void scale_tables(const float L[16], const float t[15], float s, float a[16], float T[15]) {
    for (int k = 0; k < 16; ++k) a[k] = L[k] * s;
    for (int k = 0; k < 15; ++k) T[k] = t[k] * s;
}

/* Block absmax: s = max |x_i| over the valid elements (exact). */
static float block_absmax(const float* x, int n) {
    float s = 0.0f;
    for (int i = 0; i < n; ++i) {
        float ax = fabsf(x[i]);
        if (ax > s) s = ax;
    }
    return s;
}

/* ZE-EDEN calibration of one block (listing page Abstract: after its RTN
 * codes are chosen, the block's second-moment scale is recalibrated; Table 2
 * EDEN column).  Reading: the EDEN
 * scale |y|^2 / <y, yhat> (Vargaftik et al., EDEN, ICML 2022) with
 * y = v * (1/s) and yhat = L[q], folded into the stored block scale.
 * Sums run in one fixed order: 32 groups of 4 consecutive elements, each
 * summed left to right; then an xor-butterfly over the group index with
 * offsets 1, 2, 4, 8, 16 (p_g <- p_g + p_{g^o}); the result is p_0.
 * Padding elements of a partial block contribute exact zeros.  A block
 * whose scale is below the smallest normal FP32 (including zero) keeps s. */
static float eden_block_scale(const float* v, const uint8_t* q, int n, const float L[16], float s) {
    if (!(s >= 0x1p-126f)) return s;
    float rho = 1.0f / s;
    float pa[32], pb[32];
    for (int g = 0; g < 32; ++g) {
        float sa = 0.0f, sb = 0.0f;
        for (int i = 0; i < 4; ++i) {
            int e = 4 * g + i;
            float y = (e < n) ? v[e] * rho : 0.0f;
            float yh = (e < n) ? L[q[e]] : 0.0f;
            float ta = y * y;
            float tb = y * yh;
            if (i == 0) { sa = ta; sb = tb; }
            else { sa = sa + ta; sb = sb + tb; }
        }
        pa[g] = sa;
        pb[g] = sb;
    }
    for (int o = 1; o < 32; o <<= 1) {
        float na[32], nb[32];
        for (int g = 0; g < 32; ++g) {
            na[g] = pa[g] + pa[g ^ o];
            nb[g] = pb[g] + pb[g ^ o];
        }
        memcpy(pa, na, sizeof pa);
        memcpy(pb, nb, sizeof pb);
    }
    float A = pa[0], B = pb[0];
    if (B == 0.0f) return 0.0f;
    return s * (A / B);
}

/* Nibble packing: element 2k in the low nibble of byte k, 2k+1 in the high
 * nibble (reading: the pages only say "packed 4-bit"). */
static void pack_block(const uint8_t* codes, uint8_t* out) {
    for (int k = 0; k < OB / 2; ++k) out[k] = (uint8_t)((codes[2 * k] & 15u) | ((codes[2 * k + 1] & 15u) << 4));
}
static int code_at(const uint8_t* packed, int64_t e) {
    uint8_t b = packed[e >> 1];
    return (e & 1) ? (b >> 4) : (b & 15u);
}

/* ------------------------------------------------------------------ */
/* Public block-level helpers (used by the oracle's own tests)          */
/* ------------------------------------------------------------------ */

/* Quantise one block x[0..n) with rule `rule` against levels L (thresholds
 * t for RTN).  words[i] are the 32-bit draws for SR rules; c2/eps define
 * r for the Update rules (lr etc. do not enter).  Writes codes[0..n) and
 * returns the block scale s = max|x|. */
float oracle_quant_block_r(const float L[16], const float t[15], const float* x, int n, int rule,
                           const uint32_t* words, float rb, float rc, float eps, uint8_t* codes) {
    scal_t sc;
    memset(&sc, 0, sizeof sc);
    sc.c2 = rc;
    sc.eps = eps;
    sc.rb = rb;
    sc.rc = rc;
    float s = block_absmax(x, n);
    float a[16], T[15];
    scale_tables(L, t, s, a, T);
    for (int i = 0; i < n; ++i) {
        int c = 0;
        switch (rule) {
            case RULE_STATE_RTN: c = rule_state_rtn(T, x[i]); break;
            case RULE_STATE_SR: c = rule_state_sr(a, x[i], oracle_uniform(words[i])); break;
            case RULE_UPDATE_RTN: c = rule_update_rtn(a, x[i], rule_r(x[i], &sc), &sc); break;
            case RULE_UPDATE_SR: c = rule_update_sr(a, x[i], rule_r(x[i], &sc), oracle_uniform(words[i]), &sc); break;
            default: c = 0;
        }
        codes[i] = (uint8_t)c;
    }
    return s;
}

/* As oracle_quant_block_r with the Update rules in the same-step space
 * r(x) = 1 / (sqrt(x) * c2 + eps). */
float oracle_quant_block(const float L[16], const float t[15], const float* x, int n, int rule,
                         const uint32_t* words, float c2, float eps, uint8_t* codes) {
    return oracle_quant_block_r(L, t, x, n, rule, words, 1.0f, c2, eps, codes);
}

float oracle_eden_scale(const float* v, const uint8_t* q, int n, const float L[16], float s) {
    return eden_block_scale(v, q, n, L, s);
}

/* Dequantise: value = L[q] * s. */
void oracle_dequant(const float L[16], const uint8_t* packed, const float* scales, int64_t numel, float* out) {
    for (int64_t e = 0; e < numel; ++e) out[e] = L[code_at(packed, e)] * scales[e / OB];
}

/* One unquantised AdamW step in FP32 with the same per-element op sequence
 * as the quantised step (the reduction the method must match when
 * quantisation is removed). */
void oracle_adamw_fp32(float* theta, const float* grad, float* m, float* v, int64_t n, float lr, float beta1,
                       float beta2, float eps, float wd, int64_t t) {
    scal_t s = make_scalars(lr, beta1, beta2, eps, wd, t);
    for (int64_t i = 0; i < n; ++i) {
        float g = grad[i];
        float m1 = fmaf(s.beta1, m[i], s.omb1 * g);
        float v1 = fmaf(s.beta2, v[i], s.omb2 * (g * g));
        float r = precond(v1, &s);
        theta[i] = theta[i] * s.decay - s.step_size * (m1 * r);
        m[i] = m1;
        v[i] = v1;
    }
}

/* ------------------------------------------------------------------ */
/* Factored second moment (AReno docs, State representation): rank >= 2  */
/* tensors viewed as [rows, cols] keep row means R and column means C of */
/* g^2 as exponential averages; vhat_ij = R_i * C_j / mean_i(R_i).        */
/* Sums run in double (exact per-term g^2 of BF16 inputs), rounded once. */
/* Under data parallelism the same page adds each rank's row and column  */
/* sums over the group, and R and C are updated from the totals:         */
/* factored_partials adds one shard's sums, factored_finalize applies    */
/* the update from the sums over the whole parameter.                    */
/* ------------------------------------------------------------------ */
static double clipped(uint16_t h, float clip) {
    float g = bf16_to_f32(h);
    return (double)(clip != 1.0f ? g * clip : g);
}

/* Adds the squares of the shard's (clipped) gradients to row_sums[rows] and
 * col_sums[cols].  The shard holds the elements [fbase, fbase + numel) of
 * the row-major [rows, cols] matrix; grad[e] is its element fbase + e.
 * Elements are visited in row-major order, so each row's and each column's
 * terms are added in order of increasing column and row index. */
static void factored_partials(const uint16_t* grad, int64_t numel, int64_t fbase, int64_t cols, float clip,
                              double* row_sums, double* col_sums) {
    for (int64_t e = 0; e < numel; ++e) {
        int64_t ge = fbase + e;
        double g = clipped(grad[e], clip);
        row_sums[ge / cols] += g * g;
        col_sums[ge % cols] += g * g;
    }
}

/* R_i <- fma(beta2, R_i, (1-beta2) * FP32(row_sums[i] / cols)), C_j likewise
 * with rows; then mean(R) in double, rounded once. */
static void factored_finalize(const scal_t* s, const double* row_sums, const double* col_sums, int64_t rows,
                              int64_t cols, float* R, float* C, float* rbar_out) {
    for (int64_t i = 0; i < rows; ++i) {
        float mean = (float)(row_sums[i] / (double)cols);
        R[i] = fmaf(s->beta2, R[i], s->omb2 * mean);
    }
    for (int64_t j = 0; j < cols; ++j) {
        float mean = (float)(col_sums[j] / (double)rows);
        C[j] = fmaf(s->beta2, C[j], s->omb2 * mean);
    }
    double acc = 0.0;
    for (int64_t i = 0; i < rows; ++i) acc += R[i];
    *rbar_out = (float)(acc / (double)rows);
}

/* ------------------------------------------------------------------ */
/* The fused step on one parameter tensor.                              */
/* ------------------------------------------------------------------ */
typedef struct {
    float* param;             /* FP32 master, numel (in/out) */
    const uint16_t* grad;     /* BF16 gradient, numel (in) */
    uint16_t* param_bf16;     /* BF16 copy, numel (out), may be NULL */
    uint8_t* m_codes;         /* ceil(numel/128)*64 bytes */
    float* m_scale;           /* ceil(numel/128) */
    uint8_t* v_codes;         /* packed v or NULL (factored rank >= 2) */
    float* v_scale;
    float* v_row;             /* factored R[rows] or NULL */
    float* v_col;             /* factored C[cols] or NULL */
    int64_t numel, rows;
    uint64_t elem_offset;     /* global index of element 0 (Philox counter) */
    uint32_t tensor_id, flags;
} oracle_tensor;

typedef struct {
    float nf4[16], nf4_t[15];
    float dyn4[16], dyn4_t[15];
    float dyn4nz[16], dyn4nz_t[15];
    float sdyn4[16], sdyn4_t[15];
    float lin4nz[16], lin4nz_t[15];
} oracle_codebooks;

/* Global gradient-norm clipping (AReno docs "State representation": norm and
 * clipping run directly on the BF16 gradient shards; listing page: global
 * gradient-clipping events).  Reading: torch.nn.utils.clip_grad_norm_ with
 * the 2-norm, clip = min(1, max_norm * (1 / (norm + 1e-6))), every operation
 * in FP32 as torch rounds it, norm = sqrt of the sum of squares below, and
 * the factor multiplies the FP32 value of each BF16 gradient inside the step
 * (before the moments, the factored statistics included).
 * The sum of squares runs in one canonical FP32 order:
 *   tile (elements [256 i, 256 i + 256) of a tensor; missing elements 0): lane
 *     l = 0..31 sums the squares of its 8 elements 8l..8l+7 pairwise,
 *     ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)); then an xor butterfly over the
 *     lanes with offsets 1, 2, 4, 8, 16; the result is lane 0's value;
 *   tensor: the tile sums in a complete binary tree over the tile index
 *     (padded with zeros to a power of two, adjacent pairs at every level);
 *   list: the tensor sums left to right in list order, from 0.           */
static float tile_sqsum(const uint16_t* grad, int64_t numel, int64_t tile) {
    float q[32];
    for (int l = 0; l < 32; ++l) {
        float sq[8];
        for (int k = 0; k < 8; ++k) {
            int64_t e = tile * 256 + 8 * l + k;
            float g = (e < numel) ? bf16_to_f32(grad[e]) : 0.0f;
            sq[k] = g * g;
        }
        q[l] = ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));
    }
    for (int o = 1; o < 32; o <<= 1) {
        float nq[32];
        for (int l = 0; l < 32; ++l) nq[l] = q[l] + q[l ^ o];
        memcpy(q, nq, sizeof q);
    }
    return q[0];
}

static float pow2_tree(float* a, int64_t n) {
    if (n == 0) return 0.0f;
    int64_t p = 1;
    while (p < n) p <<= 1;
    for (int64_t w = 1; w < p; w <<= 1)
        for (int64_t i = 0; i + w < p; i += 2 * w) {
            float x = (i < n) ? a[i] : 0.0f;
            float y = (i + w < n) ? a[i + w] : 0.0f;
            if (i < n) a[i] = x + y;
        }
    return a[0];
}

float oracle_grad_sqnorm(const oracle_tensor* T, int n, float* scratch) {
    float total = 0.0f;
    for (int t = 0; t < n; ++t) {
        int64_t tiles = (T[t].numel + 255) / 256;
        for (int64_t i = 0; i < tiles; ++i) scratch[i] = tile_sqsum(T[t].grad, T[t].numel, i);
        total = total + pow2_tree(scratch, tiles);
    }
    return total;
}

/* torch's coefficient: max_norm times the FP32 reciprocal of (norm + 1e-6)
 * (two roundings), clamped above at 1; a NaN norm gives a NaN factor. */
float oracle_clip_factor(float sqnorm, float max_norm) {
    float norm = sqrtf(sqnorm);
    float rcp = 1.0f / (norm + 1e-6f);
    float c = max_norm * rcp;
    return (c >= 1.0f) ? 1.0f : c;
}

/* A factored parameter stepped as one shard: its [rows, cols] matrix, the
 * shard's first element fbase in it, and the sums of squares over every
 * shard (NULL: the shard is the whole tensor, fbase 0, cols = numel / rows,
 * and the sums are its own). */
typedef struct {
    int64_t cols, fbase;
    const double *row_sums, *col_sums;
} shard_t;

static int step_tensor(const oracle_codebooks* cb, const oracle_tensor* T, float lr, float beta1, float beta2,
                       float eps, float wd, int64_t step, uint64_t seed, int recipe, uint32_t call_flags,
                       float clip, const shard_t* sh);

int oracle_step_tensor(const oracle_codebooks* cb, const oracle_tensor* T, float lr, float beta1, float beta2,
                       float eps, float wd, int64_t step, uint64_t seed, int recipe, uint32_t call_flags) {
    return step_tensor(cb, T, lr, beta1, beta2, eps, wd, step, seed, recipe, call_flags, 1.0f, NULL);
}

/* The step with gradients scaled by `clip` (oracle_clip_factor). */
int oracle_step_tensor_clip(const oracle_codebooks* cb, const oracle_tensor* T, float lr, float beta1, float beta2,
                            float eps, float wd, int64_t step, uint64_t seed, int recipe, uint32_t call_flags,
                            float clip) {
    return step_tensor(cb, T, lr, beta1, beta2, eps, wd, step, seed, recipe, call_flags, clip, NULL);
}

/* Data-parallel factored statistics, one rank's part: adds the sums of
 * (clip g)^2 of the shard T (elements [T->elem_offset, T->elem_offset +
 * T->numel) of its parameter's row-major [T->rows, cols] matrix) into
 * row_sums[T->rows] and col_sums[cols]. */
void oracle_factored_partials(const oracle_tensor* T, int64_t cols, float clip, double* row_sums,
                              double* col_sums) {
    factored_partials(T->grad, T->numel, (int64_t)T->elem_offset, cols, clip, row_sums, col_sums);
}

/* The step of one shard T of a factored parameter (T->rows rows, `cols`
 * columns; v_row and v_col hold the whole parameter's R and C), with R and C
 * updated from the sums over all shards (the sums every rank's
 * oracle_factored_partials added up); element e of the shard reads R and C
 * at matrix position T->elem_offset + e.  A tensor that is not factored is
 * stepped as by oracle_step_tensor_clip. */
int oracle_step_tensor_sums(const oracle_codebooks* cb, const oracle_tensor* T, int64_t cols, const double* row_sums,
                            const double* col_sums, float lr, float beta1, float beta2, float eps, float wd,
                            int64_t step, uint64_t seed, int recipe, uint32_t call_flags, float clip) {
    shard_t sh = {cols, (int64_t)T->elem_offset, row_sums, col_sums};
    return step_tensor(cb, T, lr, beta1, beta2, eps, wd, step, seed, recipe, call_flags, clip, &sh);
}

static int step_tensor(const oracle_codebooks* cb, const oracle_tensor* T, float lr, float beta1, float beta2,
                       float eps, float wd, int64_t step, uint64_t seed, int recipe, uint32_t call_flags,
                       float clip, const shard_t* sh) {
    if (step < 1 || T->numel < 0) return -1;
    scal_t s = make_scalars(lr, beta1, beta2, eps, wd, step);
    const int factored = (recipe == OR_FACTORED) && (T->flags & OT_FACTORED);
    /* Listing page Table 2: the LM-head first moment switches to SR in the
     * final phase under ZIP-SR and ZE-EDEN; the TorchAO baseline keeps RTN. */
    const int m_sr = ((T->flags & OT_LM_HEAD) && (call_flags & OS_LM_HEAD_SR_ACTIVE) && recipe != OR_TORCHAO) ||
                     (call_flags & OS_M_SR_ALL);
    const int v_update_rtn = (recipe == OR_ZIP_SR) && (call_flags & OS_V_UPDATE_RTN);
    const int v_next_r = (recipe == OR_ZIP_SR) && (call_flags & OS_V_NEXT_R);
    if (v_next_r) {
        float hn[6];
        oracle_host_scalars(lr, beta1, beta2, wd, step + 1, hn);
        s.rb = beta2;
        s.rc = hn[1];
    }
    int64_t cols = 0, fbase = 0;
    float rbar = 0.0f;
    if (factored && sh == NULL) {
        if (T->rows < 1 || T->numel % T->rows) return -3;
        cols = T->numel / T->rows;
        double* rs = (double*)calloc((size_t)(T->rows + cols + 1), sizeof(double));
        if (!rs) return -2;
        factored_partials(T->grad, T->numel, 0, cols, clip, rs, rs + T->rows);
        factored_finalize(&s, rs, rs + T->rows, T->rows, cols, T->v_row, T->v_col, &rbar);
        free(rs);
    } else if (factored) {
        if (T->rows < 1 || sh->cols < 1 || sh->fbase < 0 || sh->fbase + T->numel > T->rows * sh->cols) return -3;
        cols = sh->cols;
        fbase = sh->fbase;
        factored_finalize(&s, sh->row_sums, sh->col_sums, T->rows, cols, T->v_row, T->v_col, &rbar);
    }
    /* Listing page Table 2: ZIP-SR v in Dyn4, ZE-EDEN v in Dyn4-NZ, TorchAO
     * v in Lin4-NZ and m in SDyn4; AReno docs: factored 1-D v excludes zero. */
    const float* Lv = (recipe == OR_ZIP_SR) ? cb->dyn4 : (recipe == OR_TORCHAO) ? cb->lin4nz : cb->dyn4nz;
    const float* tv = (recipe == OR_ZIP_SR) ? cb->dyn4_t : (recipe == OR_TORCHAO) ? cb->lin4nz_t : cb->dyn4nz_t;
    const float* Lm = (recipe == OR_TORCHAO) ? cb->sdyn4 : cb->nf4;
    const float* tm = (recipe == OR_TORCHAO) ? cb->sdyn4_t : cb->nf4_t;

    int64_t nblocks = (T->numel + OB - 1) / OB;
    for (int64_t b = 0; b < nblocks; ++b) {
        int64_t e0 = b * OB;
        int n = (int)((T->numel - e0) < OB ? (T->numel - e0) : OB);
        float m1[OB], v1[OB], r[OB];
        /* 1-3: dequantise, moment recurrences, update and BF16 copy. */
        float sm_old = T->m_scale[b];
        float sv_old = factored ? 0.0f : T->v_scale[b];
        for (int i = 0; i < n; ++i) {
            int64_t e = e0 + i;
            float g = bf16_to_f32(T->grad[e]);
            if (clip != 1.0f) g = g * clip;
            float m = Lm[code_at(T->m_codes, e)] * sm_old;
            float mm = fmaf(s.beta1, m, s.omb1 * g);
            float vv;
            if (factored) {
                int64_t ri = (fbase + e) / cols, cj = (fbase + e) % cols;
                vv = (rbar == 0.0f) ? 0.0f : (T->v_row[ri] * T->v_col[cj]) / rbar;
            } else {
                float v = Lv[code_at(T->v_codes, e)] * sv_old;
                vv = fmaf(s.beta2, v, s.omb2 * (g * g));
            }
            float rr = precond(vv, &s);
            float th = T->param[e] * s.decay - s.step_size * (mm * rr);
            T->param[e] = th;
            if (T->param_bf16) T->param_bf16[e] = f32_to_bf16_rne(th);
            m1[i] = mm;
            v1[i] = vv;
            r[i] = rr;
        }
        /* 4-6: m requantisation (NF4, State-RTN; State-SR on the LM head
         * during its SR phase: listing page Table 2 note). */
        uint8_t qm[OB], qv[OB];
        memset(qm, 0, sizeof qm);
        memset(qv, 0, sizeof qv);
        float sm = block_absmax(m1, n);
        float am[16], Tm[15];
        scale_tables(Lm, tm, sm, am, Tm);
        for (int i = 0; i < n; ++i) {
            if (m_sr) {
                uint32_t w = oracle_draw(seed, (uint32_t)step, T->tensor_id, T->elem_offset + (uint64_t)(e0 + i), OP_M_SR);
                qm[i] = (uint8_t)rule_state_sr(am, m1[i], oracle_uniform(w));
            } else {
                qm[i] = (uint8_t)rule_state_rtn(Tm, m1[i]);
            }
        }
        pack_block(qm, T->m_codes + b * (OB / 2));
        T->m_scale[b] = sm;
        if (factored) continue;
        /* 7-8: v requantisation. */
        float sv = block_absmax(v1, n);
        float av[16], Tv[15];
        scale_tables(Lv, tv, sv, av, Tv);
        if (recipe == OR_ZIP_SR && v_next_r)
            for (int i = 0; i < n; ++i) r[i] = rule_r(v1[i], &s);
        if (recipe == OR_ZIP_SR && v_update_rtn) {
            for (int i = 0; i < n; ++i) qv[i] = (uint8_t)rule_update_rtn(av, v1[i], r[i], &s);
        } else if (recipe == OR_ZIP_SR) {
            for (int i = 0; i < n; ++i) {
                uint32_t w = oracle_draw(seed, (uint32_t)step, T->tensor_id, T->elem_offset + (uint64_t)(e0 + i), OP_V_SR);
                qv[i] = (uint8_t)rule_update_sr(av, v1[i], r[i], oracle_uniform(w), &s);
            }
        } else {
            for (int i = 0; i < n; ++i) qv[i] = (uint8_t)rule_state_rtn(Tv, v1[i]);
            if (recipe == OR_ZE_EDEN) sv = eden_block_scale(v1, qv, n, Lv, sv);
        }
        pack_block(qv, T->v_codes + b * (OB / 2));
        T->v_scale[b] = sv;
    }
    return 0;
}

/* Vectorised draw helper for tests: words[i] for idx0 + i. */
void oracle_draws(uint64_t seed, uint32_t step, uint32_t tensor_id, uint64_t idx0, uint32_t purpose, int64_t n,
                  uint32_t* words) {
    for (int64_t i = 0; i < n; ++i) words[i] = oracle_draw(seed, step, tensor_id, idx0 + (uint64_t)i, purpose);
}

void oracle_bf16_round(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(x[i]);
}
