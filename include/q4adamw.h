/*
 * q4adamw.h -- C ABI of the B300 (sm_103a) fused 4-bit AdamW optimizer step.
 *
 * The method: "Rounding in Preconditioner Space: Redesigning 4-bit AdamW
 * Optimizer-State Quantization" (Li et al., arXiv:2610.12444).  Its listing
 * page's Abstract and Table 2 define the two recipes:
 *   ZIP-SR  -- NF4 first moment (RTN), zero-inclusive dynamic-exponent 4-bit
 *              second moment with stochastic rounding whose probabilities are
 *              chosen in preconditioner space r = 1/(sqrt(v_hat)+eps);
 *   ZE-EDEN -- NF4 first moment (RTN), zero-excluding dynamic-exponent 4-bit
 *              second moment (RTN) with an EDEN rescale of each block;
 * both round the LM head's first moment stochastically on the NF4 grid in
 * the last tenth of the training steps (Table 2 note).  The AReno docs page "4-bit AdamW",
 * section "State representation", adds the factored mode (Adafactor row and
 * column means over [shape[0], -1] for rank >= 2, packed zero-excluding v for
 * 1-D tensors) and fixes the 128-element parameter-local block.  The news page
 * (paragraph 4) fixes the storage: 4-bit codes plus one FP32 scale per block
 * and moment, 1.0625 bytes/param for m+v.
 *
 * Conventions for every entry point:
 *   - All buffers are owned by the caller.  Device pointers point to memory
 *     of the current CUDA device; `stream` is a cudaStream_t (NULL = legacy
 *     default stream).  The library allocates no device memory.
 *   - Calls that take a stream are asynchronous with respect to the host:
 *     they validate, enqueue kernels and return.  A kernel error surfaces at
 *     the caller's next synchronisation.
 *   - Every call returns a q4_status; none aborts, throws or exits.  On any
 *     validation error nothing is enqueued.  Q4_ECUDA means a CUDA runtime
 *     call failed; q4adamw_last_cuda_error() returns its cudaError_t.
 *   - Blocks are 128 consecutive elements of one tensor in row-major flat
 *     order; block b covers elements [128b, min(128b+128, numel)).
 *   - Codes are packed two per byte: element 2k of a block in the low nibble
 *     of byte k, element 2k+1 in the high nibble.  Code c indexes the
 *     codebook's levels sorted ascending.  Each block owns 64 code bytes even
 *     when it is partial; nibbles past numel are written as 0.
 */
#ifndef Q4ADAMW_H
#define Q4ADAMW_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4ADAMW_BLOCK 128        /* elements per quantisation block */
#define Q4ADAMW_STATE_FORMAT 1   /* version of the state layout below */
#define Q4ADAMW_MAGIC 0x57413451u /* "Q4AW" little-endian */

typedef enum q4_status {
    Q4_OK = 0,
    Q4_EINVAL = -1,     /* null pointer where one is required, n < 0, step < 1,
                           beta outside [0,1), eps <= 0, non-finite lr / wd */
    Q4_EALIGN = -2,     /* a pointer violates the alignment stated below */
    Q4_ESHAPE = -3,     /* numel < 0; factored tensor with rows < 1 or rows
                           not dividing numel; elem_offset not a multiple of
                           128 */
    Q4_ERECIPE = -4,    /* unknown recipe or codebook id */
    Q4_EVERSION = -5,   /* state header does not match this library/recipe */
    Q4_ECUDA = -6,      /* a CUDA runtime call failed */
    Q4_EWORKSPACE = -7  /* workspace NULL, too small or not 256-B aligned */
} q4_status;

typedef enum q4_recipe {
    Q4_RECIPE_ZIP_SR = 0,   /* listing page Table 2, row "ZIP-SR 4-bit" */
    Q4_RECIPE_ZE_EDEN = 1,  /* listing page Table 2, row "ZE-EDEN 4-bit" */
    Q4_RECIPE_FACTORED = 2, /* AReno docs, State representation */
    Q4_RECIPE_TORCHAO = 3   /* listing page Table 2, row "TorchAO 4-bit": the
                               paper's baseline -- SDyn4 State-RTN first moment
                               (LM head included), Lin4-NZ State-RTN second
                               moment, no EDEN */
} q4_recipe;

/* Per-tensor flags (q4adamw_tensor_t.flags). */
#define Q4_T_LM_HEAD  0x1u  /* this tensor is the LM head: its m uses NF4
                               stochastic rounding while Q4_LM_HEAD_SR_ACTIVE */
#define Q4_T_FACTORED 0x2u  /* rank >= 2 tensor: under Q4_RECIPE_FACTORED its v
                               is the factored row/column form; ignored by the
                               other recipes */

/* Per-call flags (q4adamw_step). */
#define Q4_LM_HEAD_SR_ACTIVE 0x1u /* the final 10% phase of the schedule: the
                                     caller sets it when step > 0.9 * total
                                     (no effect under Q4_RECIPE_TORCHAO) */
#define Q4_M_SR_ALL 0x2u          /* rounding variant (listing page Tables 1,
                                     11): State-SR for the first moment of
                                     every tensor, in every phase */
#define Q4_V_UPDATE_RTN 0x4u      /* rounding variant (Table 1): Update-RTN in
                                     place of Update-SR for the second moment;
                                     Q4_RECIPE_ZIP_SR only, Q4_EINVAL otherwise */
#define Q4_V_NEXT_R 0x8u          /* rounding variant (Table 1 evaluates the
                                     preconditioner at step t+1 with a gradient
                                     of order eps): the second moment's Update
                                     rule (SR, or RTN with Q4_V_UPDATE_RTN)
                                     works in r'(q) = 1/(sqrt(beta2 q) *
                                     c2(t+1) + eps), c2(t+1) = 1/sqrt(1 -
                                     beta2^(t+1)), instead of the same-step r;
                                     Q4_RECIPE_ZIP_SR only.  Runs the general
                                     (slower) kernel path. */

/*
 * One parameter tensor and its optimizer state.  All pointers are device
 * pointers owned by the caller.
 *   param       FP32 master weights, numel.                    in/out, 16-B aligned
 *   grad        BF16 gradient (raw bits), numel.               in,     16-B aligned
 *   param_bf16  BF16 copy of the updated weights, numel.       out,    16-B aligned, may be NULL
 *   m_codes     NF4 codes of m, ceil(numel/128)*64 bytes.      in/out, 16-B aligned
 *   m_scale     FP32 absmax scale of m per block.              in/out, 4-B aligned
 *   v_codes     dynamic-exponent codes of v, as m_codes.       in/out, NULL for factored tensors
 *   v_scale     FP32 scale of v per block.                     in/out, NULL for factored tensors
 *   v_row       factored row factor R, rows floats.            in/out, factored tensors only
 *   v_col       factored column factor C, numel/rows floats.   in/out, factored tensors only
 *   numel       number of elements (0 allowed: nothing to do)
 *   rows        shape[0] of the tensor ([rows, numel/rows] view); 1 for 1-D
 *   elem_offset global index of element 0 within the full parameter, for a
 *               data-parallel shard; a multiple of 128.  Random draws depend
 *               only on (seed, step, tensor_id, elem_offset + index).
 *   tensor_id   stable id of the parameter (a random-draw key component)
 *   flags       Q4_T_* bits
 */
typedef struct q4adamw_tensor {
    float* param;
    const uint16_t* grad;
    uint16_t* param_bf16;
    uint8_t* m_codes;
    float* m_scale;
    uint8_t* v_codes;
    float* v_scale;
    float* v_row;
    float* v_col;
    int64_t numel;
    int64_t rows;
    uint64_t elem_offset;
    uint32_t tensor_id;
    uint32_t flags;
} q4adamw_tensor_t;

/*
 * State header: what a checkpoint of the 4-bit state must carry so that it is
 * resumed only by this optimizer in this representation (AReno docs,
 * "Requirements and errors": a checkpoint of the 4-bit state can be resumed
 * by this optimizer alone, and states of older formats are rejected).  Host
 * memory.
 */
typedef struct q4adamw_header {
    uint32_t magic;       /* Q4ADAMW_MAGIC */
    uint32_t format;      /* Q4ADAMW_STATE_FORMAT */
    uint32_t recipe;      /* q4_recipe */
    uint32_t block;       /* Q4ADAMW_BLOCK */
    int64_t n_tensors;
    int64_t numel_total;
} q4adamw_header_t;

/* State-format version of this library (Q4ADAMW_STATE_FORMAT). */
int q4adamw_version(void);

/* Static, NUL-terminated description of a q4_status (never NULL). */
const char* q4adamw_strerror(int status);

/* cudaError_t of the most recent Q4_ECUDA on the calling thread (0 if none). */
int q4adamw_last_cuda_error(void);

/*
 * Storage of the persistent 4-bit state (AReno docs "Requirements and
 * errors": adam4_quantized_state_bytes, adam4_scale_metadata_bytes,
 * adam4_total_bytes).  Host-only; reads numel/rows/flags of t[0..n) only.
 *   quantized   code bytes of m and v (64 B per block and packed moment)
 *   scale_meta  FP32 block scales, plus R and C floats of factored tensors
 *   total       quantized + scale_meta
 * For packed tensors whose numel is a multiple of 128 this is exactly
 * 1.0625 bytes/param (news page, paragraph 4).  Any output pointer may be NULL.
 */
int q4adamw_state_bytes(const q4adamw_tensor_t* t, int n, int recipe, int64_t* quantized, int64_t* scale_meta,
                        int64_t* total);

/* Device workspace q4adamw_step, q4adamw_step_clip and q4adamw_grad_sqnorm
 * need for this tensor list (host-only).  The workspace holds the descriptor
 * table, for factored tensors the partial row/column sums, and the
 * gradient-norm partial sums.  It must be 256-B aligned. */
int q4adamw_workspace_bytes(const q4adamw_tensor_t* t, int n, int recipe, int64_t* bytes);

/*
 * Zero-initialise the state of t[0..n): codes, scales and factored R, C.
 * A zero scale decodes every code to 0, so the first step starts from
 * m = v = 0 as AdamW does.  If header_out is not NULL it is filled for
 * recipe.  Asynchronous on stream.
 */
int q4adamw_state_init(const q4adamw_tensor_t* t, int n, int recipe, q4adamw_header_t* header_out, void* stream);

/* Q4_OK if h was written by q4adamw_state_init of this state format for
 * recipe; Q4_EVERSION otherwise; Q4_EINVAL if h is NULL.  Host-only. */
int q4adamw_header_check(const q4adamw_header_t* h, int recipe);

/*
 * One fused 4-bit AdamW step over the tensor list t[0..n), step number
 * `step` (1-based), on `stream`.
 *
 * Per element (FP32, each operation correctly rounded; news page paragraph 2
 * and listing page Abstract for AdamW with bias correction and decoupled
 * weight decay):
 *   m  = NF4[qm] * s_m;   v = V[qv] * s_v      (factored: R_i*C_j / mean(R))
 *   m' = fma(beta1, m, (1-beta1) * g);   v' = fma(beta2, v, (1-beta2) * g*g)
 *   r  = 1 / (sqrt(v') * c2 + eps),  c2 = 1/sqrt(1 - beta2^step)
 *   param' = param * (1 - lr*wd) - (lr / (1 - beta1^step)) * (m' * r)
 *   param_bf16 = round-to-nearest-even(param')
 * Per 128-block: new scales s = max|m'|, max v'; m requantised NF4 RTN
 * (LM head with Q4_LM_HEAD_SR_ACTIVE: NF4 state-space stochastic rounding);
 * v requantised per recipe (ZIP-SR: Dyn4 with preconditioner-space SR;
 * ZE-EDEN: Dyn4-NZ RTN and the EDEN scale |y|^2/<y,yhat> folded into s_v;
 * factored: 1-D tensors Dyn4-NZ RTN, rank >= 2 tensors update R and C).
 * Stochastic rounding draws Philox4x32-10 keyed by (seed, step, tensor_id,
 * elem_offset + element index); results do not depend on launch geometry.
 *
 * workspace: device memory of at least q4adamw_workspace_bytes() bytes,
 * 256-B aligned, not used concurrently by another call.  The host tensor
 * array t is read during the call only.  Tensors must not overlap.
 * Each call uploads its descriptor table to the workspace with one
 * cudaMemcpyAsync from a pageable host buffer that the next call on the same
 * thread reuses; the call is not designed for CUDA graph capture.
 */
int q4adamw_step(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps, float weight_decay,
                 int64_t step, uint64_t seed, int recipe, uint32_t flags, void* workspace, int64_t workspace_bytes,
                 void* stream);
/* (flags: any bit outside Q4_LM_HEAD_SR_ACTIVE | Q4_M_SR_ALL | Q4_V_UPDATE_RTN |
 * Q4_V_NEXT_R, or Q4_V_UPDATE_RTN / Q4_V_NEXT_R with a recipe other than
 * ZIP-SR, returns Q4_EINVAL.) */

/*
 * Global gradient-norm clipping (AReno docs "4-bit AdamW", section "State
 * representation": the norm is taken, and the clip applied, on the BF16
 * gradients themselves, shard by shard), in two calls on one stream:
 *
 * q4adamw_grad_sqnorm writes to *sqnorm (one device float, 4-B aligned,
 * caller-owned) the FP32 sum of squares of the BF16 gradients of t[0..n):
 * per tensor, recursive pairwise summation of the squares (the tensor padded
 * with zeros to a power of two, adjacent pairs added at every level), then
 * the tensor sums added left to right from 0.  The result does not depend on
 * launch geometry.  Reads grad and numel of each tensor only (grad 16-B
 * aligned, may be NULL when numel is 0).  workspace as for q4adamw_step
 * (q4adamw_workspace_bytes covers both calls; the calls must not overlap on
 * it).  A data-parallel caller sums *sqnorm over the ranks (for instance an
 * all-reduce) before the step.
 *
 * q4adamw_step_clip is q4adamw_step with every FP32 gradient first multiplied
 * by clip = min(1, max_grad_norm * (1 / (sqrt(*sqnorm) + 1e-6))), each
 * operation correctly rounded in FP32 -- the coefficient of PyTorch's
 * clip_grad_norm_ for the 2-norm.  The factor applies before the moments and
 * the factored statistics.  *sqnorm is read on the device when the step runs.
 * max_grad_norm must be finite and > 0 (else Q4_EINVAL); sqnorm NULL is
 * Q4_EINVAL, misaligned Q4_EALIGN.  A NaN sum of squares gives NaN updates.
 */
int q4adamw_grad_sqnorm(const q4adamw_tensor_t* t, int n, float* sqnorm, void* workspace, int64_t workspace_bytes,
                        void* stream);
int q4adamw_step_clip(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                      float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags,
                      float max_grad_norm, const float* sqnorm, void* workspace, int64_t workspace_bytes,
                      void* stream);

/*
 * Data-parallel shards of factored parameters (AReno docs "4-bit AdamW",
 * section "State representation": under data parallelism each rank's sums
 * of g^2 over rows and over columns are added over the group, and only the
 * totals enter the exponential update of R and C).  Each rank passes its own shards; a shard of a
 * factored parameter i is the elements [elem_offset, elem_offset + numel)
 * of the parameter's row-major matrix [rows, full_numel[i] / rows]
 * (elem_offset a multiple of 128, as for every tensor; numel may be 0).
 * v_row and v_col hold the whole parameter's R (rows floats) and C
 * (full_numel[i] / rows floats): every rank keeps its own copy and updates
 * it identically.  full_numel NULL means every tensor is whole (matrix
 * offset 0, full_numel = numel).  Tensors that are not factored in the
 * recipe ignore full_numel and step as in q4adamw_step.
 *
 * One step is three calls per rank:
 *   1. q4adamw_dp_factored_sums writes this rank's FP32 sums of g^2 (g
 *      multiplied first by the clip factor when sqnorm is not NULL, as in
 *      q4adamw_step_clip) into sums: for each factored tensor in list order,
 *      its rows' sums (rows floats; 0 for rows the shard does not touch),
 *      then its columns' sums (cols floats).  Within a shard the order of
 *      the additions is fixed (as in the single-call step).
 *   2. The caller adds the sums buffers of all ranks (an all-reduce, SUM).
 *      Every rank must pass the same factored tensors in the same order, a
 *      shard with no element included, so that the buffers line up.
 *   3. q4adamw_dp_step updates R_i <- beta2 R_i + (1-beta2) (S_i / cols) and
 *      C_j likewise (S_j / rows) from the added sums, forms mean(R) and runs
 *      the step of this rank's shards with vhat = R_i C_j / mean(R) at each
 *      element's matrix position.
 * With one rank (each parameter one shard) the result equals q4adamw_step
 * (q4adamw_step_clip) bit for bit.
 *
 * q4adamw_dp_state_init: q4adamw_state_init for such a shard list (codes and
 * scales of the shard, the whole R and C of each factored parameter, also for
 * an empty shard).
 * q4adamw_dp_sums_floats: floats of the sums buffer (host-only).
 * q4adamw_dp_workspace_bytes: the workspace both device calls need
 * (host-only; 256-B aligned, not shared with a concurrent call).
 * Errors: as q4adamw_step; Q4_ESHAPE when full_numel[i] is negative or not a
 * multiple of rows, or the shard does not fit in the matrix; Q4_EINVAL for a
 * NULL sums (with factored tensors present) or NULL v_row / v_col of a
 * factored shard, also an empty one; Q4_EALIGN for a misaligned sums.
 */
int q4adamw_dp_state_init(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                          q4adamw_header_t* header_out, void* stream);
int q4adamw_dp_sums_floats(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel, int64_t* floats);
int q4adamw_dp_workspace_bytes(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                               int64_t* bytes);
int q4adamw_dp_factored_sums(const q4adamw_tensor_t* t, int n, int recipe, const int64_t* full_numel,
                             float max_grad_norm, const float* sqnorm, float* sums, void* workspace,
                             int64_t workspace_bytes, void* stream);
int q4adamw_dp_step(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                    float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags,
                    const int64_t* full_numel, const float* sums, float max_grad_norm, const float* sqnorm,
                    void* workspace, int64_t workspace_bytes, void* stream);

/*
 * Optional check of the gradients (a counter the step itself does not keep, so
 * that the step pays nothing for it): writes to *count (one device uint64, 8-B
 * aligned, caller-owned) the number of BF16 gradient elements of t[0..n) that
 * are NaN, +inf or -inf (exponent bits all ones).  One pass over the gradients
 * (2 bytes per element).  Reads grad and numel of each tensor only (grad 16-B
 * aligned, may be NULL when numel is 0).  workspace as for q4adamw_step
 * (q4adamw_workspace_bytes covers this call; the calls must not overlap on
 * it).  Asynchronous on stream.  The pages have no counterpart: a caller may
 * use it to skip the step of a batch whose gradients overflowed.  Q4_EINVAL
 * for NULL count or n < 0, Q4_EALIGN, Q4_ESHAPE, Q4_EWORKSPACE as for
 * q4adamw_grad_sqnorm.
 */
int q4adamw_grad_nonfinite(const q4adamw_tensor_t* t, int n, uint64_t* count, void* workspace,
                           int64_t workspace_bytes, void* stream);

/*
 * The stochastic-rounding draws of the step, for checking and reproducing its
 * rounding: writes to out[0..n) (device, 4-B aligned) the 32-bit Philox4x32-10
 * words that q4adamw_step draws for elements idx0 .. idx0+n-1 (global element
 * index = elem_offset + index in the tensor) of tensor tensor_id at step
 * `step` with `seed`; purpose 0 is the first moment's State-SR, 1 the second
 * moment's Update-SR.  The uniform is u = (word >> 8) * 2^-24.  Asynchronous
 * on stream.  Q4_EINVAL for n < 0, out NULL with n > 0, step outside
 * [1, 2^32), purpose > 15; Q4_EALIGN for a misaligned out.
 */
int q4adamw_draws(uint64_t seed, int64_t step, uint32_t tensor_id, uint64_t idx0, uint32_t purpose, int64_t n,
                  uint32_t* out, void* stream);

/*
 * Status word of the most recent q4adamw_step that used `workspace`
 * (synchronises `stream`, then reads 4 bytes of the workspace).  0 means the
 * step ran to completion.  Bit 0 (Q4_STATUS_STAGE_TIMEOUT) means a warp of the
 * step kernel waited about a second for its staged input without seeing it
 * arrive and stopped; the tensors it had not reached are not updated.  Other
 * bits are reserved.  Returns Q4_EINVAL for NULL pointers, Q4_EWORKSPACE for a
 * misaligned workspace, Q4_ECUDA if the copy fails.
 */
#define Q4_STATUS_STAGE_TIMEOUT 0x1u
int q4adamw_step_status(const void* workspace, uint32_t* status, void* stream);

/*
 * Limit, in SM clock cycles, of the step kernel's bounded wait for a staged
 * tile, for the calling thread's subsequent q4adamw_step, q4adamw_step_clip
 * and q4adamw_step_noalloc calls (a per-thread setting; host-only).  0
 * restores the default of 2,000,000,000 cycles (about one second at the
 * B300's 2.03 GHz).  A warp whose wait exceeds the limit sets
 * Q4_STATUS_STAGE_TIMEOUT in the step's status word, then waits, with the
 * default limit, for the copies it still has in flight and stops; the tiles
 * it had not computed keep their previous values.  A short limit exists to
 * exercise that path: the data always arrives, only later.  The pages have
 * no counterpart (the staging and its bounded wait are this library's
 * design).  Returns Q4_EINVAL for a negative value.
 */
int q4adamw_set_stage_wait_limit(int64_t cycles);

/*
 * Decode the state of one tensor into FP32 device buffers of numel floats
 * (either may be NULL): m_out = NF4[qm]*s_m; v_out = V[qv]*s_v for packed v
 * (V = Dyn4 for ZIP-SR, Lin4-NZ for TorchAO, Dyn4-NZ otherwise; m in SDyn4 for TorchAO) or R_i*C_j/mean(R) for a factored
 * tensor.  Asynchronous on stream.
 */
int q4adamw_dequant_state(const q4adamw_tensor_t* t, int recipe, float* m_out, float* v_out, void* stream);

/*
 * q4adamw_step without a caller workspace.  The paper has no counterpart: this
 * exists for callers that cannot allocate device memory for the workspace --
 * code running inside another framework's memory budget (its caching
 * allocator already holds the device memory, so a cudaMalloc would fail or
 * fragment it) and code on a latency-critical path where cudaMalloc's implicit
 * device synchronisation is not acceptable.  It allocates nothing: the
 * workspace is a statically allocated device array of
 * Q4ADAMW_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps until
 * the process exits.  Arguments and results are those of q4adamw_step.
 *   - A tensor list whose workspace (q4adamw_workspace_bytes) exceeds
 *     Q4ADAMW_NOALLOC_SCRATCH_BYTES is rejected with Q4_EWORKSPACE before any
 *     device work.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress).  A failed lookup returns Q4_ECUDA.
 *   - All calls share the one array and it keeps the previous call's contents;
 *     every byte a step reads from it is written earlier in the same step, so
 *     nothing needs clearing.  Calls whose GPU work overlaps (different streams
 *     without ordering, or different host threads) race on the array: order them.
 */
#define Q4ADAMW_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)
int q4adamw_step_noalloc(const q4adamw_tensor_t* t, int n, float lr, float beta1, float beta2, float eps,
                         float weight_decay, int64_t step, uint64_t seed, int recipe, uint32_t flags, void* stream);

/*
 * Status word of the most recent q4adamw_step_noalloc on the current device
 * (the counterpart of q4adamw_step_status for the static scratch, whose
 * device address callers never see): synchronises `stream`, then reads the
 * word; 0 means the step ran to completion, Q4_STATUS_STAGE_TIMEOUT as for
 * q4adamw_step_status.  Like the step, it shares the one array: read it on
 * the stream of the call it reports on, before the next noalloc call.  Q4_EINVAL
 * for a NULL status, Q4_ECUDA if the address lookup or the copy fails.
 */
int q4adamw_step_noalloc_status(uint32_t* status, void* stream);

/*
 * The library's own codebook tables (host-only).  which: 0 = NF4, 1 = Dyn4
 * (zero-inclusive), 2 = Dyn4-NZ (zero-excluding), 3 = SDyn4 (signed dynamic
 * exponent), 4 = Lin4-NZ (k/16, k = 1..16).  levels: 16 ascending FP32
 * levels; thresholds: the 15 FP32 RTN decision points (rounded double
 * midpoints).  Either pointer may be NULL.
 */
int q4adamw_codebook(int which, float* levels, float* thresholds);

#ifdef __cplusplus
}
#endif

#endif /* Q4ADAMW_H */
