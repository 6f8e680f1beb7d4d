/*
 * flce.h -- C ABI of the GB300 (sm_103a) fused linear cross entropy library.
 *
 * Two operations:
 *
 *  flce_fwd_bwd  Fused linear cross entropy (FLCE): the lm_head projection
 *                z = H W^T (+ b) fused with softmax cross entropy (ignore_index,
 *                reduction none / sum / mean) and its backward (grad_hidden,
 *                grad_weight, grad_bias), chunked over tokens so the [N, V]
 *                logits never exist.  Defined by "Peak Performance, Minimized
 *                Memory: Optimizing torchtune's performance with torch.compile
 *                & Liger Kernel", section "Introduction to Liger Kernel",
 *                Figure 1 "Fused Linear Cross Entropy" and its four steps
 *                (flatten, project chunk by chunk, partial loss + chunk
 *                logits gradient, hidden gradient + accumulated head
 *                gradient); call shape from the liger-kernel 0.0.1 -> 0.1.1
 *                PyPI diff, README "Compose Your Own Model" (weight, input,
 *                target, then backward).
 *
 *  ce_fwd_bwd    Cross entropy on materialised logits [N, V]: loss and the
 *                logits gradient in one call, the gradient optionally
 *                written over the logits.  Defined by the same README,
 *                "Kernels" list, CrossEntropy item (PyTorch CrossEntropyLoss
 *                semantics, loss and gradient computed together, in-place
 *                replacement of the input); logits dtypes and the reduction /
 *                ignore contract from DeepSpeed PR #8540 (optional Liger
 *                vocab-parallel CE backend), "Changes" and "Real-device
 *                validation".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer to memory the caller owns.  The
 *    library never allocates, frees or synchronises; all work is enqueued on
 *    `stream` (a cudaStream_t; NULL is the legacy default stream) and runs
 *    asynchronously.  Outputs are valid once the stream reaches the call.
 *  - Matrices are row-major and contiguous.  bf16 is IEEE bfloat16; results
 *    stored as bf16 are rounded to nearest even.
 *  - Host-checkable faults (NULL required pointer, bad enum, bad shape or
 *    alignment, workspace too small) return an error code BEFORE anything is
 *    enqueued.  FLCE_ERR_CUDA means a launch failed (cudaGetLastError).
 *  - Device-detected faults never trap.  They are OR-ed as bits into the
 *    device status word: a target outside [0, V) that is not ignore_index sets
 *    FLCE_STATUS_BIT_TARGET_RANGE and that row is treated as ignored; a
 *    pipeline wait that exceeded its time limit sets FLCE_STATUS_BIT_TIMEOUT
 *    and that call's outputs are undefined.  The status word is `status_dev`
 *    when given (never cleared by the library), else the first 4 bytes of the
 *    workspace (cleared at the start of each call).
 *  - Calls that share a workspace must not overlap in time (same stream, or
 *    ordered by events).
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here so the header needs no CUDA. */
typedef struct CUstream_st* flce_stream_t;

typedef enum {
  FLCE_REDUCTION_NONE = 0, /* per-row losses [N]                      */
  FLCE_REDUCTION_SUM = 1,  /* sum over valid rows, scalar             */
  FLCE_REDUCTION_MEAN = 2  /* sum / number of valid rows (NaN if 0)   */
} flce_reduction_t;

/* FLCE_DTYPE_FP32_ROUNDED: fp32 FLCE operands rounded to bf16 once (the
 * fast mode of flce_fwd_bwd_typed); not a logits type. */
typedef enum {
  FLCE_DTYPE_BF16 = 0,
  FLCE_DTYPE_FP32 = 1,
  FLCE_DTYPE_FP16 = 2,
  FLCE_DTYPE_FP32_ROUNDED = 3
} flce_dtype_t;

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad enum       */
  FLCE_ERR_UNSUPPORTED = 2,  /* dtype or layout not handled (e.g. H % 8)    */
  FLCE_ERR_WORKSPACE = 3,    /* workspace NULL/too small/misaligned         */
  FLCE_ERR_CUDA = 4,         /* a CUDA call or kernel launch failed         */
  FLCE_ERR_TARGET_RANGE = 5, /* value of a device status bit (see above)    */
  FLCE_ERR_TIMEOUT = 6,      /* value of a device status bit (see above)    */
  FLCE_ERR_MISALIGNED = 7    /* a pointer breaks its alignment requirement  */
} flce_status_t;

/* Bits of the device status word. */
#define FLCE_STATUS_BIT_TARGET_RANGE 0x1
#define FLCE_STATUS_BIT_TIMEOUT 0x2

/* Human-readable name of a status code (static storage, never NULL). */
const char* flce_status_string(flce_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int flce_version(void);

/* ------------------------------------------------------------------------
 * Fused linear cross entropy
 * ------------------------------------------------------------------------ */

/* Token chunk used when flce_fwd_bwd is given chunk = 0, for these sizes. */
int64_t flce_default_chunk(int64_t N, int64_t H, int64_t V);

/* Bytes of workspace flce_fwd_bwd needs for these sizes (chunk 0 = default).
 * It grows with chunk * V (the bf16 logits / grad-logits of one chunk) and
 * with N (4 bytes of per-row loss), never with N * V.  Returns 0 for invalid
 * sizes. */
size_t flce_workspace_size(int64_t N, int64_t H, int64_t V, int64_t chunk, int reduction);

/* flce_workspace_size_typed -- the workspace flce_fwd_bwd_typed needs for
 * operands of `dtype` (flce_dtype_t); 0 for an unknown dtype or invalid
 * sizes. */
size_t flce_workspace_size_typed(int dtype, int64_t N, int64_t H, int64_t V, int64_t chunk,
                                 int reduction);

/*
 * flce_fwd_bwd -- loss and gradients of cross_entropy(hidden @ weight^T + bias, target).
 *
 *  hidden        bf16 [N, H]; 16-byte aligned; H a multiple of 8 (TMA rows).
 *  weight        bf16 [V, H]; 16-byte aligned.
 *  bias          bf16 [V] or NULL (no bias).
 *  target        int64 [N]; class ids in [0, V) or ignore_index.
 *  N, H, V       tokens (>= 0), hidden size (>= 8, % 8 == 0), vocabulary (>= 1).
 *  ignore_index  targets equal to it add no loss and no gradient (checked
 *                before the range check, so it may lie inside [0, V)).
 *  reduction     flce_reduction_t.  Mean divides by the number of valid
 *                targets over all N rows.
 *  chunk         tokens per chunk (>= 1), or 0 for flce_default_chunk.
 *  grad_scale    upstream gradient g of the reduced loss; multiplies every
 *                gradient (1.0 for plain loss.backward()).
 *  grad_out_none fp32 [N] per-row upstream gradients, reduction NONE only
 *                (gradient of sum_n g * grad_out[n] * loss_n); NULL = ones.
 *  loss          fp32 output: [N] for NONE (0 for ignored rows), else [1].
 *  grad_hidden   bf16 [N, H] output (always overwritten), or NULL to skip.
 *  grad_weight   fp32 [V, H] output, 16-byte aligned, or NULL to skip.
 *  grad_bias     fp32 [V] output, or NULL to skip (must be NULL if bias is).
 *  accumulate    0: grad_weight / grad_bias are overwritten; 1: added to.
 *  n_valid_out   int32 [1] output (number of valid targets), or NULL.
 *  lse_out       fp32 [N] output: log-sum-exp of every row's logits, or NULL.
 *  target_logit_out  fp32 [N] output: z[n, target_n] for valid rows, 0 for
 *                ignored rows, or NULL.  (These two are the per-row partials
 *                a vocabulary-parallel caller would combine across shards.)
 *  workspace     device scratch of >= flce_workspace_size(...) bytes,
 *                256-byte aligned; contents on entry are ignored.
 *  status_dev    int32 device status word (see conventions), or NULL.
 *  stream        CUDA stream.
 *
 * Arithmetic: the projection runs on the tensor cores (bf16 x bf16, fp32
 * accumulation); the log-sum-exp and the target logit come from the fp32
 * accumulator; the chunk's grad-logits are rounded to bf16 before the two
 * backward products, which accumulate in fp32.
 */
flce_status_t flce_fwd_bwd(const void* hidden, const void* weight, const void* bias,
                           const int64_t* target, int64_t N, int64_t H, int64_t V,
                           int64_t ignore_index, int reduction, int64_t chunk,
                           float grad_scale, const float* grad_out_none, float* loss,
                           void* grad_hidden, float* grad_weight, float* grad_bias,
                           int accumulate, int32_t* n_valid_out, float* lse_out,
                           float* target_logit_out, void* workspace, size_t workspace_bytes,
                           int32_t* status_dev, flce_stream_t stream);

/*
 * flce_fwd_bwd_typed -- flce_fwd_bwd with the operand type given: dtype is
 *   FLCE_DTYPE_BF16          exactly flce_fwd_bwd;
 *   FLCE_DTYPE_FP16          hidden, weight, bias and grad_hidden are IEEE half;
 *   FLCE_DTYPE_FP32          hidden, weight, bias and grad_hidden are fp32,
 *                            multiplied at about fp32 accuracy (below);
 *   FLCE_DTYPE_FP32_ROUNDED  the same buffers, the operands rounded to bf16
 *                            once (the fast mode, below);
 * everything else is as in flce_fwd_bwd.  The workspace must hold
 * flce_workspace_size_typed(dtype, ...) bytes (the same as
 * flce_workspace_size for the two 16-bit types; FP32 adds bf16 hi + lo
 * copies of hidden and weight and a second plane of chunk logits,
 * FP32_ROUNDED one bf16 copy of hidden, weight and bias).  Other dtypes return
 * FLCE_ERR_UNSUPPORTED.  The logits dtypes FP32 / FP16 / BF16
 * the DeepSpeed PR #8540 description ("optional Liger vocab-parallel CE
 * backend", section "Changes") validates carry over to the fused form here.
 *
 * Arithmetic with fp16: fp16 x fp16 on the tensor cores with fp32
 * accumulation; the chunk logits are kept in fp16, and the chunk's
 * grad-logits are stored in fp16 divided by the part of the gradient scale
 * common to all rows (g / n_valid for MEAN, g for SUM, g * max|grad_out| for
 * NONE), so they lie in [-1, 1] rather than underflowing fp16's range; the
 * two backward products multiply that factor back in fp32.  grad_bias is
 * summed from the fp32 grad-logits.
 *
 * Arithmetic with FP32: hidden and weight are split once per call into bf16
 * hi = round(x) and lo = round(x - hi) (nearest, ties to even), and every
 * product is formed on the tensor cores as hi.hi + hi.lo + lo.hi with fp32
 * accumulation (the dropped lo.lo term is below 2^-16 of each product), at
 * a third of the bf16 tensor rate; the bias is added in fp32; the chunk
 * logits are kept exactly (both halves of their fp32 bits), their gradient
 * is formed in fp32 and split the same way for the two backward products;
 * grad_hidden is written from the fp32 accumulator.
 *
 * Arithmetic with FP32_ROUNDED: hidden, weight and bias are rounded to bf16
 * (to nearest, ties to even) into the workspace once per call and the bf16
 * path runs on those copies, so the loss and grad_weight / grad_bias equal
 * the bf16 entry point's on the rounded inputs; grad_hidden is written from
 * the fp32 accumulator without the bf16 rounding.  This is the rate of the
 * bf16 path at its precision, for callers whose fp32 tensors are master
 * copies of a mixed-precision step.
 */
flce_status_t flce_fwd_bwd_typed(int dtype, const void* hidden, const void* weight, const void* bias,
                                 const int64_t* target, int64_t N, int64_t H, int64_t V,
                                 int64_t ignore_index, int reduction, int64_t chunk,
                                 float grad_scale, const float* grad_out_none, float* loss,
                                 void* grad_hidden, float* grad_weight, float* grad_bias,
                                 int accumulate, int32_t* n_valid_out, float* lse_out,
                                 float* target_logit_out, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, flce_stream_t stream);

/* ------------------------------------------------------------------------
 * Cross entropy on materialised logits
 * ------------------------------------------------------------------------ */

/* Bytes of workspace ce_fwd_bwd needs (per-row losses and counters). */
size_t ce_workspace_size(int64_t N, int64_t V, int dtype, int reduction);

/*
 * ce_fwd_bwd -- loss and grad_logits of cross_entropy(logits, target).
 *
 *  logits        [N, V] of `dtype` (FLCE_DTYPE_BF16, FLCE_DTYPE_FP16 or FLCE_DTYPE_FP32).
 *  grad_logits   [N, V] of `dtype` output: scale_n * (softmax - onehot), 0 for
 *                ignored rows.  May equal `logits` (in place: the logits are
 *                consumed) or be a separate buffer (logits left unchanged),
 *                or NULL (loss only).  Partial overlap is not allowed.
 *  target        int64 [N].
 *  ignore_index, reduction, grad_scale, grad_out_none, loss: as flce_fwd_bwd.
 *  workspace     >= ce_workspace_size(...) bytes, 256-byte aligned; contents
 *                on entry are ignored.  One workspace serves one call at a
 *                time (calls on different streams need their own).
 *  status_dev, stream: as flce_fwd_bwd.
 *
 * With 16-byte aligned logits / grad_logits pointers every row length of at
 * least 32 bytes runs on 16-byte vectors (a row that is not a whole number
 * of vectors is handled through its aligned covering range, touching no
 * neighbouring row's elements); otherwise an element-by-element path runs.
 * With N <= 16384 and the vector forms the call is a single kernel launch
 * (no separate counting pass); otherwise a small counting kernel runs
 * first.
 */
flce_status_t ce_fwd_bwd(const void* logits, int dtype, void* grad_logits, const int64_t* target,
                         int64_t N, int64_t V, int64_t ignore_index, int reduction,
                         float grad_scale, const float* grad_out_none, float* loss,
                         void* workspace, size_t workspace_bytes, int32_t* status_dev,
                         flce_stream_t stream);

/* ------------------------------------------------------------------------
 * Vocabulary-parallel building blocks
 * ------------------------------------------------------------------------
 * When the vocabulary is split across shards (tensor parallelism: the
 * vocabulary-parallel cross entropy and the fused lm_head + vocabulary-
 * parallel CE that never builds the [S, B, V/tp] logits -- "Native
 * Liger-Kernel integration in Megatron-LM", PR table and Roadmap item 2;
 * DeepSpeed PR #8540 "Changes"), shard s holds vocabulary ids
 * [vocab_offset, vocab_offset + V_shard).  The cross entropy needs, per row,
 * the log-sum-exp over the whole vocabulary and the target logit; the caller
 * combines the shards' partials (for example with an all-reduce):
 *     lse = M + log(sum_s exp(lse_s - M)),  M = max_s lse_s
 *     z_t = sum_s zt_s              (zt_s is 0 unless shard s holds the target)
 * and then lets every shard form its own gradients from the combined values
 * and per-row scales row_scale[n] = d(reduced loss)/d(loss_n) (0 for ignored
 * rows), which the caller also forms (it knows the global valid count, the
 * reduction and the upstream gradient).  The loss is lse - z_t per row.
 * Targets are global ids; ignore_index marks ignored rows.
 */

/* Bytes of workspace for flce_vp_forward / flce_vp_backward on a chunk of C rows. */
size_t flce_vp_workspace_size(int64_t C, int64_t H, int64_t V_shard);

/* FLCE on one vocabulary shard, forward part, for one chunk of C tokens:
 * projects hidden [C, H] with weight_shard [V_shard, H] (+ bias_shard) into
 * the workspace (bf16) and writes per row lse_shard (fp32 logits), lse16_shard
 * (their bf16 roundings; combine it the same way for the gradient) and
 * target_logit_shard.  The workspace must then be passed, unchanged, to
 * flce_vp_backward for the same chunk.  Alignment and H as flce_fwd_bwd. */
flce_status_t flce_vp_forward(const void* hidden, const void* weight_shard, const void* bias_shard,
                              const int64_t* target, int64_t C, int64_t H, int64_t V_shard,
                              int64_t vocab_offset, int64_t ignore_index, float* lse_shard,
                              float* lse16_shard, float* target_logit_shard, void* workspace,
                              size_t workspace_bytes, int32_t* status_dev, flce_stream_t stream);

/* FLCE on one vocabulary shard, backward part: with lse16 [C] combined over
 * all shards and row_scale [C], forms the shard's logits gradient in the
 * workspace, then grad_hidden_partial (fp32 [C, H], overwritten; the caller
 * sums it over shards), grad_weight_shard (fp32 [V_shard, H]) and
 * grad_bias_shard (fp32 [V_shard]); accumulate = 1 adds to the latter two.
 * Any of the three outputs may be NULL. */
flce_status_t flce_vp_backward(const void* hidden, const void* weight_shard, const int64_t* target,
                               int64_t C, int64_t H, int64_t V_shard, int64_t vocab_offset,
                               int64_t ignore_index, const float* lse16, const float* row_scale,
                               float* grad_hidden_partial, float* grad_weight_shard,
                               float* grad_bias_shard, int accumulate, void* workspace,
                               size_t workspace_bytes, int32_t* status_dev, flce_stream_t stream);

/* Cross entropy on a vocabulary shard of materialised logits [N, V_shard]:
 * per-row partials lse_shard and target_logit_shard.  No workspace. */
flce_status_t ce_vp_partials(const void* logits, int dtype, const int64_t* target, int64_t N,
                             int64_t V_shard, int64_t vocab_offset, int64_t ignore_index,
                             float* lse_shard, float* target_logit_shard, int32_t* status_dev,
                             flce_stream_t stream);

/* ... and the shard's gradient from the combined lse [N] and row_scale [N]:
 * grad = row_scale * (softmax - onehot), written to grad_logits (may equal
 * logits).  No workspace. */
flce_status_t ce_vp_backward(const void* logits, int dtype, void* grad_logits, const int64_t* target,
                             int64_t N, int64_t V_shard, int64_t vocab_offset, int64_t ignore_index,
                             const float* lse, const float* row_scale, int32_t* status_dev,
                             flce_stream_t stream);

/* ------------------------------------------------------------------------
 * Cross entropy on logits without any caller-provided scratch
 * ------------------------------------------------------------------------ */

/* Largest N accepted by ce_fwd_bwd_noalloc. */
#define FLCE_NOALLOC_MAX_ROWS 65536

/*
 * ce_fwd_bwd_noalloc -- the computation of ce_fwd_bwd for callers that cannot
 * allocate device memory or hand over a workspace: for example a plugin whose
 * enqueue step may not allocate, a process whose device memory belongs to
 * another allocator, or a loop that cannot afford cudaMalloc's implicit
 * synchronisation.  The pages have no counterpart; it is an integration aid.
 *
 * Its scratch (256 bytes plus 4 bytes per row) is a fixed device array inside
 * the library, sized for FLCE_NOALLOC_MAX_ROWS rows (about 256 KiB, held by
 * every GPU that loads the library until the process exits).  Arguments are
 * those of ce_fwd_bwd without the workspace; N > FLCE_NOALLOC_MAX_ROWS returns
 * FLCE_ERR_UNSUPPORTED before anything is enqueued.  The entry point calls
 * no allocating routine (no cudaMalloc or cudaFree, no workspace).  Device
 * memory does appear once per device context when the CUDA runtime loads the
 * library's module (the array and the kernels' code; with lazy module
 * loading, the default, this happens at the first call and at the first
 * launch of each kernel): make one warm-up call per device outside any
 * region that must not allocate.
 *
 * The first call on a device context looks the array's device address up (a
 * CUDA runtime query with that device current; again after cudaDeviceReset,
 * whose new context holds the array elsewhere); make that first call before
 * any stream capture.  All calls share the one array: calls that may overlap
 * on the GPU (unordered streams) race and must be serialised by the caller.
 * With status_dev NULL no status is reported.  Like ce_fwd_bwd, a call with
 * N <= 16384 and the vector forms is a single kernel launch.
 */
flce_status_t ce_fwd_bwd_noalloc(const void* logits, int dtype, void* grad_logits,
                                 const int64_t* target, int64_t N, int64_t V,
                                 int64_t ignore_index, int reduction, float grad_scale,
                                 const float* grad_out_none, float* loss, int32_t* status_dev,
                                 flce_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics (no counterpart on the pages)
 * ------------------------------------------------------------------------ */

/* Time limit of every pipeline wait inside the kernels, in nanoseconds of
 * %globaltimer (default 2e9).  Applies to calls enqueued afterwards. */
void flce_set_wait_timeout_ns(uint64_t timeout_ns);

/* Enqueues a kernel whose pipeline wait can never be satisfied: after
 * timeout_ns it must give up, set FLCE_STATUS_BIT_TIMEOUT in *status_dev and
 * return.  Checks the failure path of the bounded waits without faulting. */
flce_status_t flce_selftest_wait_timeout(int32_t* status_dev, uint64_t timeout_ns,
                                         flce_stream_t stream);

/* Kernel timing: while enabled, every kernel the library enqueues is
 * bracketed by a pair of CUDA events on its stream (the library creates up
 * to `capacity` pairs once).  flce_profile_read synchronises on the recorded
 * events and returns, for each recorded launch, its kernel id (below) and
 * duration in ms; returns the number written (<= max).  Not thread-safe. */
enum {
  FLCE_KERNEL_COUNT_TARGETS = 0,
  FLCE_KERNEL_GEMM_FWD = 1,
  FLCE_KERNEL_ROW_FINALIZE = 2,
  FLCE_KERNEL_GRAD_LOGITS = 3,
  FLCE_KERNEL_GEMM_BWD = 4,
  FLCE_KERNEL_LOSS_REDUCE = 5,
  FLCE_KERNEL_CE_ROWS = 6,
  FLCE_KERNEL_ZERO = 7,
  FLCE_KERNEL_BIAS_REDUCE = 8,
  FLCE_KERNEL_GH_REDUCE = 9
};
const char* flce_kernel_name(int kernel_id);
flce_status_t flce_profile_enable(int capacity);
void flce_profile_disable(void);
int flce_profile_read(int* kernel_ids, float* ms, int max);

#ifdef __cplusplus
}
#endif
#endif /* FLCE_H_ */
