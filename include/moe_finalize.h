/*
 * moe_finalize.h -- C ABI of the GB300 (sm_103a) MoE finalize library
 * (libmoe_finalize.so).
 *
 * Three operations:
 *
 *   moe_finalize_rmsnorm  -- flashinfer.comm.tp_moe_finalize_rmsnorm (API
 *     page: description and parameter list).  Per token t, gather the
 *     unweighted GEMM2 rows selected by expanded_idx_to_permuted_idx[t, k],
 *     scale each by its routing weight, reduce in FP32, apply RMSNorm with
 *     gain norm_weight + gain_center (before or after the RMS), write BF16.
 *
 *   beam_moe_finalize     -- vllm.models.beam.nvidia.moe_finalize,
 *     beam_moe_finalize (docstring and source).  Per live token, reduce a
 *     token-major [capacity, top_k, hidden] block in FP32, round to BF16,
 *     multiply by routed_scale and round to BF16 again, optionally apply a
 *     post-RMSNorm, write BF16.
 *
 *   beam_moe_finalize_norm_residual_norm -- the same page's function of that
 *     name: the Beam finalize, then a residual add and the next RMSNorm, in one
 *     kernel (the residual step is a reading of the pages; see its comment).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device (or managed) memory of the
 *     current device; the caller owns all of them.  The library allocates no
 *     memory and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  No host synchronisation, no cross-stream ordering:
 *     when switching streams, order the work with events, as the API page
 *     requires of its own operation.
 *   - Arguments are validated on the host before anything is launched.  On a
 *     non-MF_OK return nothing was launched, except MF_ERR_CUDA, which reports
 *     the launch error.
 *   - A token count of zero is a no-op that returns MF_OK (pointers unchecked),
 *     as the Beam wrapper skips the native call when the output has no rows.
 *   - Outputs must not alias inputs (one exception: the residual op's hidden
 *     output may be its residual buffer).
 *   - Kernel waits are bounded (about two seconds of wall time); a wait that
 *     gives up sets MF_ERR_DEVICE_TIMEOUT in the device status word, which
 *     mf_device_status() reads.  After such a timeout the outputs of that call
 *     and of any later kernel on the context are unspecified: the CTA that
 *     gave up waits once more (also bounded) for its copies in flight, but if
 *     that wait gives up too, a bulk copy may still land in shared memory that
 *     another CTA then uses.  Discard the results and the CUDA context.
 *   - The first call on a device sets kernel attributes; make it before any
 *     CUDA graph capture.  Captured calls replay with their arguments baked in.
 */
#ifndef MOE_FINALIZE_H
#define MOE_FINALIZE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *mf_stream_t;

typedef enum mf_status {
    MF_OK = 0,
    MF_ERR_NULL = 1,             /* a required pointer is NULL */
    MF_ERR_SHAPE = 2,            /* sizes or strides break the tensor contract */
    MF_ERR_ALIGN = 3,            /* a pointer breaks the 16-byte (or 4-byte) alignment rule */
    MF_ERR_DTYPE = 4,            /* unknown weight dtype */
    MF_ERR_UNSUPPORTED = 5,      /* hidden / top_k outside what the operation defines */
    MF_ERR_CUDA = 6,             /* CUDA runtime error (no device, launch failure, ...) */
    MF_ERR_DEVICE_TIMEOUT = 7,   /* a bounded device-side wait gave up */
    MF_ERR_INVALID = 8           /* inconsistent argument combination or unknown variant */
} mf_status;

/* Storage of the routing weights.  MF_DTYPE_PACKED_TOPK takes the producer
 * MoE's packed int32 routing words as they are: (expert_id << 16) |
 * (bits of the BF16 weight), the topk_ids format of
 * flashinfer.fused_moe.trtllm_fp8_per_tensor_scale_routed_moe (parameter
 * list); the weight is the low 16 bits read as BF16, the expert id is ignored
 * (the row comes from the index map). */
typedef enum mf_dtype {
    MF_DTYPE_BF16 = 0,
    MF_DTYPE_FP32 = 1,
    MF_DTYPE_PACKED_TOPK = 2
} mf_dtype;

/* Kernel choice.  AUTO picks by size; the others force one kernel (for
 * validation and benchmarking, as the Beam wrappers' `strategy` argument
 * forces a path).  Every variant computes the same result up to the order of
 * the sum of squares.  A variant that does not apply returns MF_ERR_INVALID. */
typedef enum mf_variant {
    MF_VARIANT_AUTO = 0,
    MF_VARIANT_TOKEN_CTA = 1,    /* one CTA per token, gathers held in registers */
    MF_VARIANT_BULK = 2,         /* one CTA per token, rows staged in shared memory by bulk copies */
    MF_VARIANT_CLUSTER = 3       /* finalize+RMSNorm only: hidden split over a cluster, DSMEM reduction */
} mf_variant;

/*
 * moe_finalize_rmsnorm -- flashinfer.comm.tp_moe_finalize_rmsnorm (API page,
 * description and parameters gemm2_permuted, expert_weights,
 * expanded_idx_to_permuted_idx, norm_weight, output, eps, gain_center,
 * weight_before_norm), on one GPU (the page's tensor-parallel workspace does
 * not apply to a single device: world size 1).
 *
 *   gemm2_permuted   device, BF16 [rows, row_stride] row-major: unweighted GEMM2
 *                    rows in physical expert order.  Columns [0, hidden) are
 *                    used; row_stride >= hidden, row_stride % 8 == 0, base
 *                    16-byte aligned (so every row start is).  May be NULL
 *                    only when rows == 0.
 *   rows             number of rows; an index i is valid iff 0 <= i < rows.
 *   expert_weights   device, [num_tokens, top_k] contiguous, BF16, FP32 or
 *                    packed int32 routing words (weights_dtype); converted to
 *                    FP32.  16-byte aligned.
 *   expanded_idx_to_permuted_idx
 *                    device, int32 [num_tokens, top_k] contiguous, 16-byte
 *                    aligned.  A negative or out-of-range index contributes
 *                    zero and its weight is never read.
 *   norm_weight      device, BF16 [hidden], 16-byte aligned.
 *   output           device, BF16 [num_tokens, hidden] contiguous, 16-byte
 *                    aligned.
 *   hidden, top_k    4096 and 8, the sizes the operation is defined for (the
 *                    specialised kernels), or any hidden in 256..8192 that is
 *                    a multiple of 256 with top_k in 1..32 (the range the Beam
 *                    wrapper accepts; one generic kernel, variant AUTO or BULK).
 *   eps              added to the mean square inside the square root.
 *   gain_center      added to norm_weight in FP32: g = float(norm_weight) + gain_center.
 *   weight_before_norm  nonzero: y = v / rms(v) with v = acc * g;
 *                    zero: y = acc / rms(acc) * g.
 *
 * For each token: acc[h] = sum over valid slots k, in ascending k, of
 * w[t,k] * gemm2[idx[t,k], h] as FP32 fused multiply-adds; rms(v) =
 * sqrt(mean_h v[h]^2 + eps) over the `hidden` columns; output = BF16(y)
 * rounded to nearest even.
 *
 * Errors: MF_ERR_SHAPE (num_tokens < 0 or above 2^27 - 1, rows < 0,
 * row_stride < hidden or not a multiple of 8), MF_ERR_UNSUPPORTED (hidden / top_k outside the sizes
 * above), MF_ERR_INVALID (TOKEN_CTA or CLUSTER for sizes other than 4096 / 8),
 * MF_ERR_NULL, MF_ERR_ALIGN, MF_ERR_DTYPE, MF_ERR_CUDA.
 */
mf_status moe_finalize_rmsnorm(const void *gemm2_permuted, int64_t rows, int64_t row_stride,
                               const void *expert_weights, mf_dtype weights_dtype,
                               const int32_t *expanded_idx_to_permuted_idx,
                               const void *norm_weight, void *output, int64_t num_tokens,
                               int32_t hidden, int32_t top_k, float eps, float gain_center,
                               int weight_before_norm, mf_stream_t stream);

/* moe_finalize_rmsnorm with an explicit kernel choice (same arguments and
 * results; every variant gives the same output bits). */
mf_status moe_finalize_rmsnorm_variant(const void *gemm2_permuted, int64_t rows,
                                       int64_t row_stride, const void *expert_weights,
                                       mf_dtype weights_dtype,
                                       const int32_t *expanded_idx_to_permuted_idx,
                                       const void *norm_weight, void *output,
                                       int64_t num_tokens, int32_t hidden, int32_t top_k,
                                       float eps, float gain_center, int weight_before_norm,
                                       mf_variant variant, mf_stream_t stream);

/*
 * beam_moe_finalize -- vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize
 * (docstring: only the output rows are reduced, with BF16 rounds kept before
 * the scale and before the norm; source: the argument assertions and the
 * native call).
 *
 *   expert_outputs   device, BF16 [capacity, top_k, hidden] contiguous,
 *                    token-major, 16-byte aligned.  Rows t >= live_tokens are
 *                    never read.
 *   capacity         first dimension of expert_outputs.
 *   expert_weights   device, FP32 [weight_rows, top_k] contiguous, 4-byte
 *                    aligned; weight_rows >= live_tokens.
 *   output           device, BF16 [live_tokens, hidden] contiguous, 16-byte
 *                    aligned.  Only these rows are written.
 *   live_tokens      0 <= live_tokens <= capacity.
 *   top_k            1 .. 32.
 *   hidden           256 .. 8192, a multiple of 256.
 *   routed_scale     multiplier applied to the BF16-rounded reduction.
 *   post_weight      device BF16 [hidden] (16-byte aligned) or NULL; needs
 *                    has_post_norm.
 *   post_eps         RMSNorm epsilon (inside the square root).
 *   has_post_norm    nonzero: apply the post-RMSNorm (unweighted when
 *                    post_weight is NULL); zero: output = v.
 *
 * For each live token: s[h] = sum_k w[t,k] * x[t,k,h] (FP32 fused
 * multiply-adds, ascending k); r = BF16(s); v = BF16(float(r) * routed_scale)
 * (FP32 product); with the norm, output = BF16(v / sqrt(mean v^2 + post_eps)
 * * post_weight), else output = v.
 *
 * Errors: MF_ERR_UNSUPPORTED (top_k or hidden out of range), MF_ERR_SHAPE
 * (live_tokens < 0, > capacity or above 2^31 - 1, weight_rows < live_tokens), MF_ERR_INVALID
 * (post_weight without has_post_norm), MF_ERR_NULL, MF_ERR_ALIGN, MF_ERR_CUDA.
 */
mf_status beam_moe_finalize(const void *expert_outputs, int64_t capacity,
                            const float *expert_weights, int64_t weight_rows, void *output,
                            int64_t live_tokens, int32_t top_k, int32_t hidden,
                            float routed_scale, const void *post_weight, float post_eps,
                            int has_post_norm, mf_stream_t stream);

/* beam_moe_finalize with an explicit kernel choice (TOKEN_CTA or BULK). */
mf_status beam_moe_finalize_variant(const void *expert_outputs, int64_t capacity,
                                    const float *expert_weights, int64_t weight_rows,
                                    void *output, int64_t live_tokens, int32_t top_k,
                                    int32_t hidden, float routed_scale, const void *post_weight,
                                    float post_eps, int has_post_norm, mf_variant variant,
                                    mf_stream_t stream);

/*
 * beam_moe_finalize_norm_residual_norm -- vllm.models.beam.nvidia.moe_finalize,
 * beam_moe_finalize_norm_residual_norm (docstring: the local tokens are
 * carried from the finalize up to the following normalisation; source: the
 * assertions and the unfused reference), on one GPU.  For each of the first
 * `tokens` rows:
 *
 *   f          = the beam_moe_finalize result for the row (above), including
 *                its optional post-RMSNorm, rounded to BF16
 *   hidden     = BF16(scale_x * f + scale_residual * residual)   FP32: one
 *                product, one fused multiply-add
 *   normalized = BF16(hidden / sqrt(mean(hidden^2) + next_eps) * next_weight)
 *                when has_next_norm (unweighted if next_weight is NULL)
 *
 * The residual step stands for the unfused reference's beam_norm_residual_norm,
 * given the finalized rows, the residual, next_weight, next_eps and scales,
 * whose body the pages do not show: this reading of it
 * (scales = (scale_x, scale_residual), (1, 1) when the caller has none) is
 * partly unpinned.
 *
 *   expert_outputs, capacity, expert_weights, weight_rows, top_k, hidden,
 *   routed_scale, post_weight, post_eps, has_post_norm: as for beam_moe_finalize,
 *                    with tokens in place of live_tokens.
 *   residual         device BF16 [tokens, hidden] contiguous, 16-byte aligned.
 *   tokens           0 <= tokens <= capacity, weight_rows >= tokens.
 *   next_weight      device BF16 [hidden] (16-byte aligned) or NULL; needs has_next_norm.
 *   hidden_out       device BF16 [tokens, hidden], 16-byte aligned; may be the
 *                    residual buffer itself (an in-place residual update).
 *   normalized_out   device BF16 [tokens, hidden], 16-byte aligned, required
 *                    when has_next_norm and NULL otherwise.
 *
 * Errors: MF_ERR_UNSUPPORTED, MF_ERR_SHAPE, MF_ERR_INVALID (a weight without
 * its norm flag, normalized_out without has_next_norm), MF_ERR_NULL,
 * MF_ERR_ALIGN, MF_ERR_CUDA.  Zero tokens: MF_OK, nothing launched.
 */
mf_status beam_moe_finalize_norm_residual_norm(
    const void *expert_outputs, int64_t capacity, const float *expert_weights, int64_t weight_rows,
    const void *residual, int64_t tokens, int32_t top_k, int32_t hidden, float routed_scale,
    const void *post_weight, float post_eps, int has_post_norm, const void *next_weight,
    float next_eps, int has_next_norm, float scale_x, float scale_residual, void *hidden_out,
    void *normalized_out, mf_stream_t stream);

/* The kernel AUTO would run for moe_finalize_rmsnorm with these sizes on the
 * calling thread's current device (MF_VARIANT_AUTO if none would run: no
 * tokens or unsupported sizes).  At 4096 / 8: the cluster kernel up to 8
 * tokens, the bulk-staged kernel from 1024; in between the register kernel
 * (MF_VARIANT_TOKEN_CTA) unless the bulk-staged kernel covers the tokens in
 * fewer waves of resident CTAs (the device's SM count times each kernel's CTAs
 * per SM).  Without a usable device the wave test is skipped.  Sizes other than
 * 4096 / 8 always run the generic bulk-staged kernel (MF_VARIANT_BULK). */
mf_variant mf_select_finalize_variant(int64_t num_tokens, int32_t hidden, int32_t top_k);

/* The kernel AUTO would run for beam_moe_finalize. */
mf_variant mf_select_beam_variant(int64_t live_tokens, int32_t top_k, int32_t hidden);

/* Name of the CUDA kernel that moe_finalize_rmsnorm_variant would launch for
 * these sizes and this variant on the calling thread's current device, for
 * diagnostics and for matching a profiler's launch list: "tp_cluster_kernel",
 * "tp_token_cta_kernel", "tp_token_bulk_kernel", "tp_token_bulk_multi_kernel"
 * (the staged kernel with several tokens per CTA, from five waves of tokens
 * up), "tp_generic_bulk_kernel", "tp_generic_bulk_multi_kernel" (other sizes
 * with several tokens per CTA, on the same rule), "tp_warp_bulk_kernel" or
 * "tp_warp_bulk_multi_kernel" (hidden 256..1024, several tokens per warp).
 * The empty string when nothing would launch (no tokens, unsupported sizes, a
 * variant that does not apply).  Static string. */
const char *mf_finalize_kernel_name(int64_t num_tokens, int32_t hidden, int32_t top_k,
                                    mf_variant variant);

/* The same for beam_moe_finalize_variant, and with nonzero `residual` for
 * beam_moe_finalize_norm_residual_norm: "beam_token_bulk_kernel",
 * "beam_token_bulk_multi_kernel" (hidden 4096..7168, several tokens per CTA:
 * the residual op from five waves of tokens up, plain Beam at small top_k or
 * where one token per CTA leaves little data in flight), "beam_warp_bulk_kernel"
 * (hidden 256..1024) or "beam_token_cta_kernel". */
const char *mf_beam_kernel_name(int64_t live_tokens, int32_t top_k, int32_t hidden,
                                mf_variant variant, int residual);

/* Human-readable name of a status code (static string). */
const char *mf_status_string(mf_status status);

/* Read the device status word of the current device after synchronising it:
 * MF_OK, or MF_ERR_DEVICE_TIMEOUT if any kernel's bounded wait gave up since
 * the word was last cleared.  Nonzero `clear` resets the word.  MF_ERR_CUDA
 * if the device cannot be reached. */
mf_status mf_device_status(int clear);

/* Failure-detection self-test: launch one block whose thread waits on an
 * mbarrier that nothing will ever complete, bounded by timeout_ns (clamped to
 * at most one second).  The wait gives up, records MF_ERR_DEVICE_TIMEOUT in
 * the device status word and the kernel returns normally; the context stays
 * usable.  Read the result with mf_device_status(). */
mf_status mf_selftest_wait_timeout(uint64_t timeout_ns, mf_stream_t stream);

/* Measurement aid, not part of the operation: the memory traffic of
 * moe_finalize_rmsnorm at hidden 4096 and top_k 8, without its arithmetic.
 * The arguments mean what they mean there (gemm2_permuted BF16 [rows,
 * row_stride]; expert_weights and expanded_idx_to_permuted_idx [num_tokens,
 * 8]; output BF16 [num_tokens, 4096], device pointers, 16-byte aligned).  One
 * CTA per token reads the token's route, copies each valid row into shared
 * memory, reads it back and stores one 4096-element output row, so the call
 * moves the same bytes as the finalize; what it stores is a bit pattern of no
 * meaning (the XOR of the words read).  Timing it beside the finalize on the
 * same buffers shows what the reduction, the norm and the finalize's kernel
 * scheduling add to the traffic itself.  Statuses and the bounded waits as
 * for moe_finalize_rmsnorm (MF_ERR_SHAPE for a row stride under 4096 or not a
 * multiple of 8, or more than 2^31 - 1 tokens). */
mf_status mf_finalize_data_movement(const void *gemm2_permuted, int64_t rows, int64_t row_stride,
                                    const void *expert_weights, mf_dtype weights_dtype,
                                    const int32_t *expanded_idx_to_permuted_idx, void *output,
                                    int64_t num_tokens, mf_stream_t stream);

/* Programmatic dependent launch (process-wide, on by default).  When on, every
 * kernel is launched with the programmatic stream serialisation attribute: it
 * may be scheduled before the previous kernel in the stream has fully
 * retired, and it waits for that kernel's completion (griddepcontrol.wait)
 * before its first global-memory access, so results are the same either way;
 * back-to-back small calls lose part of their launch gap.  The setting applies to later
 * calls; the producer MoE op exposes the same choice as enable_pdl
 * (flashinfer.fused_moe.trtllm_fp8_per_tensor_scale_routed_moe, parameter list). */
void mf_set_programmatic_launch(int enable);
int mf_get_programmatic_launch(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t mf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FINALIZE_H */
