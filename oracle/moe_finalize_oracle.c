/*
 * CPU oracle for the MoE finalize (+ RMSNorm) path and its Beam variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, `__graft_entry__.smoke()` and the CPU
 * baseline leg of `bench.py` use it.  It shares no code, header or constant
 * with the CUDA library under moe_finalize_rmsnorm_gb300/csrc/.
 *
 * It is the plain definition of the operation, one element at a time, slow
 * on purpose:
 *
 *   flashinfer.comm.tp_moe_finalize_rmsnorm (API page, description and the
 *   parameter list):
 *     acc[t,h] = sum over slots k whose index i = idx[t,k] satisfies
 *                0 <= i < rows of  w[t,k] * gemm2[i,h]        (FP32)
 *     g[h]     = float(norm_weight[h]) + gain_center          (FP32 add)
 *     weight_before_norm: v = acc * g, y = v / sqrt(mean_h v^2 + eps)
 *     otherwise:          v = acc,     y = acc / sqrt(mean_h acc^2 + eps) * g
 *     output[t,h] = bf16(y)
 *
 *   vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize (docstring and
 *   source):
 *     s[t,h] = sum_k w[t,k] * x[t,k,h]                         (FP32)
 *     r = bf16(s);  v = bf16(float(r) * routed_scale)
 *     has_norm: y = v / sqrt(mean_h v^2 + post_eps) * (post_weight or 1),
 *               output = bf16(y);  otherwise output = v
 *     only rows t < live_tokens are produced.
 *
 * Precision.  The API page fixes FP32 for the routing reduction (the rows are
 * widened to FP32 and the weighted sum stays in FP32), so the
 * reduction runs in float with slots in ascending order, one fused
 * multiply-add (C99 fmaf, single rounding) per slot.  The pages fix no
 * precision for the normalisation, so it runs in double (float64), and the
 * result is rounded once from double to BF16, round-to-nearest-even.  That
 * includes the pre-norm gain product of weight_before_norm, acc * g, which is
 * formed in double from the two FP32 values (exact there: no extra rounding).  For the
 * Beam scale, which the docstring applies to the expert reduction once it has
 * been rounded to BF16, the product is read as PyTorch's BF16 tensor times a
 * scalar: an FP32 product rounded to BF16.
 *
 *   vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize_norm_residual_norm
 *   (docstring and source): the Beam finalize above (with its optional post
 *   norm) followed, for the same live rows, by the residual step of the unfused
 *   reference, which hands the finalized rows, the residual, next_weight,
 *   next_eps and scales to beam_norm_residual_norm.  That function is not shown
 *   on the pages,
 *   so this step is PARTLY UNPINNED; it is read as
 *     hidden     = BF16(s0 * finalized + s1 * residual)   FP32: one product,
 *                  then one fused multiply-add, scales (s0, s1) = (1, 1) when
 *                  none are given
 *     normalized = BF16(hidden / sqrt(mean(hidden^2) + next_eps) * next_weight)
 *                  (float64, unweighted when next_weight is absent), only when
 *                  next_eps is given.
 *
 * Readings where the pages are silent:
 *   - eps sits inside the square root (standard RMSNorm), for both ops;
 *   - "out of range" means i >= rows (rows = gemm2_permuted.shape[0]);
 *     an invalid slot is skipped entirely: its weight is never read into the
 *     sum, so a NaN weight there has no effect;
 *   - the mean runs over the `hidden` live columns only, never the row padding;
 *   - post_weight absent with post_eps given means an unweighted RMSNorm.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared ... -lm
 * (-ffp-contract=off so that the compiler fuses nothing on its own; the only
 * fused operations are the explicit fmaf calls of the reduction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- BF16 helpers (BF16 = the upper 16 bits of an IEEE binary32) -------- */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round a double to the nearest BF16 value, ties to even, in one step.
 * BF16 keeps 8 significant bits and binary32's exponent range: the spacing of
 * BF16 values in [2^(e-1), 2^e) is 2^(e-8), and below the smallest normal
 * 2^-126 the subnormal spacing is 2^-133.  x / spacing is exact (a power of
 * two scaling), rint() in the default rounding mode rounds it to the nearest
 * integer with ties to even, and the product back is a BF16 value.  Values
 * that round to 2^128 or beyond overflow to infinity; NaN becomes the
 * canonical quiet NaN 0x7FC0.
 */
uint16_t oracle_bf16_from_double(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return 0x7FC0u;
    if (isinf(x))
        return (uint16_t)(sign | 0x7F80u);
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    int e;
    (void)frexp(ax, &e); /* ax = m * 2^e with m in [0.5, 1) */
    double spacing = ldexp(1.0, ax >= ldexp(1.0, -126) ? e - 8 : -133);
    double r = rint(x / spacing) * spacing;
    if (fabs(r) >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r; /* exact: r is a BF16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

double oracle_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

/* ---- shared pieces of both ops ------------------------------------------ */

/* acc[h] = fmaf(w, x[h], acc[h]) for h < hidden: one routing slot. */
static void accumulate_row(float *acc, const uint16_t *x, float w, int32_t hidden)
{
    for (int32_t h = 0; h < hidden; ++h)
        acc[h] = fmaf(w, bf16_bits_to_float(x[h]), acc[h]);
}

/* 1 / sqrt(mean_h v[h]^2 + eps), in double. */
static double inverse_rms(const double *v, int32_t hidden, double eps)
{
    double sum_sq = 0.0;
    for (int32_t h = 0; h < hidden; ++h)
        sum_sq += v[h] * v[h];
    return 1.0 / sqrt(sum_sq / (double)hidden + eps);
}

/*
 * tp_moe_finalize_rmsnorm for tokens [0, num_tokens).
 *
 * gemm2:        BF16 bits, `rows` rows of `row_stride` elements; columns
 *               [0, hidden) are used.
 * weights:      [num_tokens, top_k]: BF16 bits (weights_kind 0), float
 *               (weights_kind 1), or the producer MoE's packed int32 routing
 *               words (weights_kind 2): (expert_id << 16) | BF16 weight bits,
 *               the topk_ids format of trtllm_fp8_per_tensor_scale_routed_moe
 *               (parameter list); the weight is the low half.
 * idx:          [num_tokens, top_k] int32.
 * norm_weight:  BF16 bits [hidden].
 * output:       BF16 bits [num_tokens, hidden].
 * Returns 0, or -1 if the scratch row could not be allocated.
 */
int oracle_moe_finalize_rmsnorm(const uint16_t *gemm2, int64_t rows, int64_t row_stride,
                                const void *weights, int weights_kind, const int32_t *idx,
                                const uint16_t *norm_weight, uint16_t *output,
                                int64_t num_tokens, int32_t hidden, int32_t top_k,
                                float eps, float gain_center, int weight_before_norm)
{
    float *acc = (float *)malloc(sizeof(float) * (size_t)hidden);
    double *v = (double *)malloc(sizeof(double) * (size_t)hidden);
    if (!acc || !v) {
        free(acc);
        free(v);
        return -1;
    }
    for (int64_t t = 0; t < num_tokens; ++t) {
        for (int32_t h = 0; h < hidden; ++h)
            acc[h] = 0.0f;
        for (int32_t k = 0; k < top_k; ++k) {
            int64_t i = idx[t * top_k + k];
            if (i < 0 || i >= rows)
                continue; /* invalid slot: contributes nothing */
            float w;
            if (weights_kind == 1)
                w = ((const float *)weights)[t * top_k + k];
            else if (weights_kind == 2)
                w = bf16_bits_to_float(
                    (uint16_t)(((const uint32_t *)weights)[t * top_k + k] & 0xFFFFu));
            else
                w = bf16_bits_to_float(((const uint16_t *)weights)[t * top_k + k]);
            accumulate_row(acc, gemm2 + i * row_stride, w, hidden);
        }
        for (int32_t h = 0; h < hidden; ++h) {
            float g = bf16_bits_to_float(norm_weight[h]) + gain_center; /* FP32 add */
            v[h] = weight_before_norm ? (double)acc[h] * (double)g : (double)acc[h];
        }
        double r = inverse_rms(v, hidden, (double)eps);
        for (int32_t h = 0; h < hidden; ++h) {
            double y;
            if (weight_before_norm) {
                y = v[h] * r;
            } else {
                float g = bf16_bits_to_float(norm_weight[h]) + gain_center;
                y = v[h] * r * (double)g;
            }
            output[t * hidden + h] = oracle_bf16_from_double(y);
        }
    }
    free(acc);
    free(v);
    return 0;
}

/*
 * beam_moe_finalize for tokens [0, live_tokens).
 *
 * expert_outputs: BF16 bits [capacity, top_k, hidden], token-major.
 * weights:        float [>= live_tokens, top_k].
 * post_weight:    BF16 bits [hidden] or NULL (unweighted norm).
 * output:         BF16 bits [live_tokens, hidden]; nothing past it is touched.
 * Returns 0, or -1 if the scratch row could not be allocated.
 */
int oracle_beam_moe_finalize(const uint16_t *expert_outputs, const float *weights,
                             uint16_t *output, int64_t live_tokens, int32_t top_k,
                             int32_t hidden, float routed_scale, const uint16_t *post_weight,
                             float post_eps, int has_post_norm)
{
    float *acc = (float *)malloc(sizeof(float) * (size_t)hidden);
    double *v = (double *)malloc(sizeof(double) * (size_t)hidden);
    if (!acc || !v) {
        free(acc);
        free(v);
        return -1;
    }
    for (int64_t t = 0; t < live_tokens; ++t) {
        for (int32_t h = 0; h < hidden; ++h)
            acc[h] = 0.0f;
        for (int32_t k = 0; k < top_k; ++k)
            accumulate_row(acc, expert_outputs + (t * top_k + k) * (int64_t)hidden,
                           weights[t * top_k + k], hidden);
        for (int32_t h = 0; h < hidden; ++h) {
            uint16_t rounded = oracle_bf16_from_double((double)acc[h]);
            float scaled = bf16_bits_to_float(rounded) * routed_scale; /* FP32 product */
            v[h] = bf16_bits_to_double(oracle_bf16_from_double((double)scaled));
        }
        if (!has_post_norm) {
            for (int32_t h = 0; h < hidden; ++h)
                output[t * hidden + h] = oracle_bf16_from_double(v[h]);
            continue;
        }
        double r = inverse_rms(v, hidden, (double)post_eps);
        for (int32_t h = 0; h < hidden; ++h) {
            double gamma = post_weight ? bf16_bits_to_double(post_weight[h]) : 1.0;
            output[t * hidden + h] = oracle_bf16_from_double(v[h] * r * gamma);
        }
    }
    free(acc);
    free(v);
    return 0;
}

/*
 * beam_moe_finalize_norm_residual_norm for tokens [0, tokens) (partly
 * unpinned: see the header comment).
 *
 * expert_outputs, weights, post_weight, post_eps, has_post_norm: as for
 * oracle_beam_moe_finalize.  residual: BF16 bits [tokens, hidden].
 * next_weight: BF16 bits [hidden] or NULL.  hidden_out: BF16 bits [tokens,
 * hidden].  normalized_out: BF16 bits [tokens, hidden], written only when
 * has_next_norm.  Returns 0, or -1 if a row buffer could not be allocated.
 */
int oracle_beam_moe_finalize_norm_residual_norm(
    const uint16_t *expert_outputs, const float *weights, const uint16_t *residual, int64_t tokens,
    int32_t top_k, int32_t hidden, float routed_scale, const uint16_t *post_weight, float post_eps,
    int has_post_norm, const uint16_t *next_weight, float next_eps, int has_next_norm,
    float scale_x, float scale_residual, uint16_t *hidden_out, uint16_t *normalized_out)
{
    uint16_t *finalized = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)hidden);
    double *v = (double *)malloc(sizeof(double) * (size_t)hidden);
    if (!finalized || !v) {
        free(finalized);
        free(v);
        return -1;
    }
    for (int64_t t = 0; t < tokens; ++t) {
        if (oracle_beam_moe_finalize(expert_outputs + t * top_k * (int64_t)hidden,
                                     weights + t * top_k, finalized, 1, top_k, hidden, routed_scale,
                                     post_weight, post_eps, has_post_norm) != 0) {
            free(finalized);
            free(v);
            return -1;
        }
        for (int32_t h = 0; h < hidden; ++h) {
            float x = bf16_bits_to_float(finalized[h]);
            float r = bf16_bits_to_float(residual[t * hidden + h]);
            float sum = fmaf(scale_residual, r, scale_x * x);
            uint16_t b = oracle_bf16_from_double((double)sum);
            hidden_out[t * hidden + h] = b;
            v[h] = bf16_bits_to_double(b);
        }
        if (!has_next_norm)
            continue;
        double rs = inverse_rms(v, hidden, (double)next_eps);
        for (int32_t h = 0; h < hidden; ++h) {
            double gamma = next_weight ? bf16_bits_to_double(next_weight[h]) : 1.0;
            normalized_out[t * hidden + h] = oracle_bf16_from_double(v[h] * rs * gamma);
        }
    }
    free(finalized);
    free(v);
    return 0;
}
