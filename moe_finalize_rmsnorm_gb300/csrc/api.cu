// C ABI of libmoe_finalize.so: argument validation, kernel selection and the
// device status word.  Declarations and the contract are in
// include/moe_finalize.h.

#include <atomic>
#include <mutex>

#include "moe_finalize.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Device status word: kernels OR mf::kStatusWaitTimeout into it when a
// bounded wait gives up.  One per device (module globals are per context).
__device__ unsigned int g_status_word;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on every device wait
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    int bulk_per_sm = 0;       // resident CTAs per SM of the staged hidden-4096 kernel
    int token_cta_per_sm = 0;  // and of the register kernel
    unsigned *status = nullptr;  // device address of g_status_word
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
std::atomic<int> g_programmatic{1};  // programmatic dependent launch, on by default

// Per-device set-up on first use: SM count, opt-in shared memory, the status
// word's device address and the kernels' attributes.
mf_status device_info(const DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                   dev) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status_word) !=
                cudaSuccess ||
            mf::prepare_tp_kernels(d.smem_optin, d.smem_per_sm) != cudaSuccess ||
            mf::prepare_beam_kernels(d.smem_per_sm) != cudaSuccess ||
            mf::tp_blocks_per_sm(&d.bulk_per_sm, &d.token_cta_per_sm) != cudaSuccess) {
            (void)cudaGetLastError();
            return MF_ERR_CUDA;
        }
        d.ready = true;
    }
    *out = &d;
    return MF_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Finalize + RMSNorm, by token count (measured on GB300):
//   <= kClusterMaxTokens  cluster kernel: a token's gather spread over 8 SMs
//                         (2.50 us per call at 1 token when the rows are in
//                         L2, as right after the producing GEMM, against
//                         2.61 us for one CTA per token);
//   <  kBulkMinTokens     register kernel (one dependent index load, then all
//                         row loads at once), unless the bulk-staged kernel,
//                         with more CTAs per SM (3 against 2 on GB300), covers
//                         the tokens in fewer waves (384 tokens: 4.15 against
//                         4.72 us; 768: 7.05 against 7.70 us; at 512, two
//                         waves each, 6.32 against 5.75 us);
//   otherwise             bulk-staged kernel (more bytes in flight per SM).
constexpr int64_t kClusterMaxTokens = 8;
constexpr int64_t kBulkMinTokens = 1024;

int64_t waves(int64_t tokens, int64_t ctas_per_wave) {
    return ctas_per_wave > 0 ? (tokens + ctas_per_wave - 1) / ctas_per_wave : 0;
}

// `d` may be null (no device information): the token-count rule alone.
mf_variant pick_tp(int64_t num_tokens, const DeviceInfo *d) {
    if (num_tokens <= 0) return MF_VARIANT_AUTO;
    if (num_tokens <= kClusterMaxTokens) return MF_VARIANT_CLUSTER;
    if (num_tokens >= kBulkMinTokens) return MF_VARIANT_BULK;
    if (d != nullptr && d->bulk_per_sm > 0 && d->token_cta_per_sm > 0 &&
        waves(num_tokens, int64_t{d->bulk_per_sm} * d->num_sms) <
            waves(num_tokens, int64_t{d->token_cta_per_sm} * d->num_sms))
        return MF_VARIANT_BULK;
    return MF_VARIANT_TOKEN_CTA;
}

// Beam: one CTA per live token with the token's block staged in shared memory.
mf_variant pick_beam(int64_t live) { return live <= 0 ? MF_VARIANT_AUTO : MF_VARIANT_BULK; }

mf_status from_launch(cudaError_t e) { return e == cudaSuccess ? MF_OK : MF_ERR_CUDA; }

}  // namespace

extern "C" {

const char *mf_status_string(mf_status s) {
    switch (s) {
        case MF_OK: return "ok";
        case MF_ERR_NULL: return "a required pointer is NULL";
        case MF_ERR_SHAPE: return "sizes or strides break the tensor contract";
        case MF_ERR_ALIGN: return "a pointer is not aligned as required";
        case MF_ERR_DTYPE: return "unknown weight dtype";
        case MF_ERR_UNSUPPORTED: return "hidden or top_k outside what the operation defines";
        case MF_ERR_CUDA: return "CUDA runtime error";
        case MF_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
        case MF_ERR_INVALID: return "inconsistent arguments or unknown variant";
    }
    return "unknown status";
}

int32_t mf_version(void) { return 100; }

void mf_set_programmatic_launch(int enable) { g_programmatic.store(enable ? 1 : 0); }

int mf_get_programmatic_launch(void) { return g_programmatic.load(); }

mf_status moe_finalize_rmsnorm_variant(const void *gemm2_permuted, int64_t rows,
                                       int64_t row_stride, const void *expert_weights,
                                       mf_dtype weights_dtype,
                                       const int32_t *expanded_idx_to_permuted_idx,
                                       const void *norm_weight, void *output,
                                       int64_t num_tokens, int32_t hidden, int32_t top_k,
                                       float eps, float gain_center, int weight_before_norm,
                                       mf_variant variant, mf_stream_t stream) {
    if (num_tokens < 0 || rows < 0) return MF_ERR_SHAPE;
    const bool specialised = hidden == mf::kTpHidden && top_k == mf::kTpTopK;
    if (!specialised && (hidden < 256 || hidden > 8192 || hidden % 256 != 0 || top_k < 1 ||
                         top_k > 32))
        return MF_ERR_UNSUPPORTED;
    if (row_stride < hidden || row_stride % 8 != 0) return MF_ERR_SHAPE;
    if (weights_dtype != MF_DTYPE_BF16 && weights_dtype != MF_DTYPE_FP32 &&
        weights_dtype != MF_DTYPE_PACKED_TOPK)
        return MF_ERR_DTYPE;
    if (variant < MF_VARIANT_AUTO || variant > MF_VARIANT_CLUSTER) return MF_ERR_INVALID;
    if (!specialised && variant != MF_VARIANT_AUTO && variant != MF_VARIANT_BULK)
        return MF_ERR_INVALID;
    if (num_tokens == 0) return MF_OK;
    if (!expert_weights || !expanded_idx_to_permuted_idx || !norm_weight || !output ||
        (rows > 0 && !gemm2_permuted))
        return MF_ERR_NULL;
    if (!aligned(gemm2_permuted, 16) || !aligned(expert_weights, 16) ||
        !aligned(expanded_idx_to_permuted_idx, 16) || !aligned(norm_weight, 16) ||
        !aligned(output, 16))
        return MF_ERR_ALIGN;
    if (num_tokens > 0x7fffffffLL / 16) return MF_ERR_SHAPE;  // grid limits of the decode kernel

    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;

    mf::TpArgs a = {};
    a.gemm2 = static_cast<const uint16_t *>(gemm2_permuted);
    a.rows = rows;
    a.ld = row_stride;
    a.weights = expert_weights;
    a.idx = expanded_idx_to_permuted_idx;
    a.norm_weight = static_cast<const uint16_t *>(norm_weight);
    a.out = static_cast<uint16_t *>(output);
    a.num_tokens = num_tokens;
    a.hidden = hidden;
    a.top_k = top_k;
    a.eps = eps;
    a.gain_center = gain_center;
    a.before = weight_before_norm ? 1 : 0;
    a.status = d->status;
    a.timeout_ns = kWaitLimitNs;
    a.programmatic = g_programmatic.load() != 0;
    const int wk = weights_dtype == MF_DTYPE_BF16   ? mf::kWeightBF16
                   : weights_dtype == MF_DTYPE_FP32 ? mf::kWeightFP32
                                                    : mf::kWeightPacked;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (!specialised)
        return from_launch(mf::launch_tp_generic(a, wk, d->smem_per_sm, d->num_sms, s));
    if (variant == MF_VARIANT_AUTO) variant = pick_tp(num_tokens, d);
    switch (variant) {
        case MF_VARIANT_CLUSTER: return from_launch(mf::launch_tp_cluster(a, wk, s));
        case MF_VARIANT_TOKEN_CTA: return from_launch(mf::launch_tp_token_cta(a, wk, s));
        case MF_VARIANT_BULK:
            return from_launch(mf::launch_tp_bulk(a, wk, d->bulk_per_sm * d->num_sms, s));
        default: return MF_ERR_INVALID;
    }
}

mf_status moe_finalize_rmsnorm(const void *gemm2_permuted, int64_t rows, int64_t row_stride,
                               const void *expert_weights, mf_dtype weights_dtype,
                               const int32_t *expanded_idx_to_permuted_idx,
                               const void *norm_weight, void *output, int64_t num_tokens,
                               int32_t hidden, int32_t top_k, float eps, float gain_center,
                               int weight_before_norm, mf_stream_t stream) {
    return moe_finalize_rmsnorm_variant(gemm2_permuted, rows, row_stride, expert_weights,
                                        weights_dtype, expanded_idx_to_permuted_idx, norm_weight,
                                        output, num_tokens, hidden, top_k, eps, gain_center,
                                        weight_before_norm, MF_VARIANT_AUTO, stream);
}

mf_status mf_finalize_data_movement(const void *gemm2_permuted, int64_t rows, int64_t row_stride,
                                    const void *expert_weights, mf_dtype weights_dtype,
                                    const int32_t *expanded_idx_to_permuted_idx, void *output,
                                    int64_t num_tokens, mf_stream_t stream) {
    if (num_tokens < 0 || rows < 0) return MF_ERR_SHAPE;
    if (row_stride < mf::kTpHidden || row_stride % 8 != 0) return MF_ERR_SHAPE;
    if (weights_dtype != MF_DTYPE_BF16 && weights_dtype != MF_DTYPE_FP32 &&
        weights_dtype != MF_DTYPE_PACKED_TOPK)
        return MF_ERR_DTYPE;
    if (num_tokens == 0) return MF_OK;
    if (!expert_weights || !expanded_idx_to_permuted_idx || !output || (rows > 0 && !gemm2_permuted))
        return MF_ERR_NULL;
    if (!aligned(gemm2_permuted, 16) || !aligned(expert_weights, 16) ||
        !aligned(expanded_idx_to_permuted_idx, 16) || !aligned(output, 16))
        return MF_ERR_ALIGN;
    if (num_tokens > 0x7fffffffLL) return MF_ERR_SHAPE;  // one CTA per token

    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;
    mf::TpArgs a = {};
    a.gemm2 = static_cast<const uint16_t *>(gemm2_permuted);
    a.rows = rows;
    a.ld = row_stride;
    a.weights = expert_weights;
    a.idx = expanded_idx_to_permuted_idx;
    a.out = static_cast<uint16_t *>(output);
    a.num_tokens = num_tokens;
    a.hidden = mf::kTpHidden;
    a.top_k = mf::kTpTopK;
    a.status = d->status;
    a.timeout_ns = kWaitLimitNs;
    a.programmatic = g_programmatic.load() != 0;
    const int wk = weights_dtype == MF_DTYPE_BF16   ? mf::kWeightBF16
                   : weights_dtype == MF_DTYPE_FP32 ? mf::kWeightFP32
                                                    : mf::kWeightPacked;
    return from_launch(
        mf::launch_tp_data_movement(a, wk, reinterpret_cast<cudaStream_t>(stream)));
}

mf_status beam_moe_finalize_variant(const void *expert_outputs, int64_t capacity,
                                    const float *expert_weights, int64_t weight_rows,
                                    void *output, int64_t live_tokens, int32_t top_k,
                                    int32_t hidden, float routed_scale, const void *post_weight,
                                    float post_eps, int has_post_norm, mf_variant variant,
                                    mf_stream_t stream) {
    if (top_k < 1 || top_k > 32) return MF_ERR_UNSUPPORTED;
    if (hidden < 256 || hidden > 8192 || hidden % 256 != 0) return MF_ERR_UNSUPPORTED;
    if (capacity < 0 || live_tokens < 0 || live_tokens > capacity || weight_rows < live_tokens)
        return MF_ERR_SHAPE;
    if (post_weight && !has_post_norm) return MF_ERR_INVALID;
    if (variant != MF_VARIANT_AUTO && variant != MF_VARIANT_TOKEN_CTA &&
        variant != MF_VARIANT_BULK)
        return MF_ERR_INVALID;
    if (live_tokens == 0) return MF_OK;
    if (!expert_outputs || !expert_weights || !output) return MF_ERR_NULL;
    if (!aligned(expert_outputs, 16) || !aligned(output, 16) || !aligned(expert_weights, 4) ||
        (post_weight && !aligned(post_weight, 16)))
        return MF_ERR_ALIGN;
    if (live_tokens > 0x7fffffffLL) return MF_ERR_SHAPE;

    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;

    mf::BeamArgs a = {};
    a.x = static_cast<const uint16_t *>(expert_outputs);
    a.weights = expert_weights;
    a.out = static_cast<uint16_t *>(output);
    a.post_weight = static_cast<const uint16_t *>(post_weight);
    a.live = live_tokens;
    a.top_k = top_k;
    a.hidden = hidden;
    a.routed_scale = routed_scale;
    a.post_eps = post_eps;
    a.has_norm = has_post_norm ? 1 : 0;
    a.status = d->status;
    a.timeout_ns = kWaitLimitNs;
    a.programmatic = g_programmatic.load() != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (variant == MF_VARIANT_AUTO) variant = pick_beam(live_tokens);
    if (variant == MF_VARIANT_BULK)
        return from_launch(mf::launch_beam_bulk(a, d->smem_per_sm, d->num_sms, false, s));
    return from_launch(mf::launch_beam_token_cta(a, s));
}

mf_status beam_moe_finalize(const void *expert_outputs, int64_t capacity,
                            const float *expert_weights, int64_t weight_rows, void *output,
                            int64_t live_tokens, int32_t top_k, int32_t hidden,
                            float routed_scale, const void *post_weight, float post_eps,
                            int has_post_norm, mf_stream_t stream) {
    return beam_moe_finalize_variant(expert_outputs, capacity, expert_weights, weight_rows, output,
                                     live_tokens, top_k, hidden, routed_scale, post_weight,
                                     post_eps, has_post_norm, MF_VARIANT_AUTO, stream);
}

mf_status beam_moe_finalize_norm_residual_norm(
    const void *expert_outputs, int64_t capacity, const float *expert_weights, int64_t weight_rows,
    const void *residual, int64_t tokens, int32_t top_k, int32_t hidden, float routed_scale,
    const void *post_weight, float post_eps, int has_post_norm, const void *next_weight,
    float next_eps, int has_next_norm, float scale_x, float scale_residual, void *hidden_out,
    void *normalized_out, mf_stream_t stream) {
    if (top_k < 1 || top_k > 32) return MF_ERR_UNSUPPORTED;
    if (hidden < 256 || hidden > 8192 || hidden % 256 != 0) return MF_ERR_UNSUPPORTED;
    if (capacity < 0 || tokens < 0 || tokens > capacity || weight_rows < tokens)
        return MF_ERR_SHAPE;
    if ((post_weight && !has_post_norm) || (next_weight && !has_next_norm) ||
        (normalized_out && !has_next_norm))
        return MF_ERR_INVALID;
    if (tokens == 0) return MF_OK;
    if (!expert_outputs || !expert_weights || !residual || !hidden_out ||
        (has_next_norm && !normalized_out))
        return MF_ERR_NULL;
    if (!aligned(expert_outputs, 16) || !aligned(residual, 16) || !aligned(hidden_out, 16) ||
        !aligned(expert_weights, 4) || (normalized_out && !aligned(normalized_out, 16)) ||
        (post_weight && !aligned(post_weight, 16)) || (next_weight && !aligned(next_weight, 16)))
        return MF_ERR_ALIGN;
    if (tokens > 0x7fffffffLL) return MF_ERR_SHAPE;

    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;

    mf::BeamArgs a = {};
    a.x = static_cast<const uint16_t *>(expert_outputs);
    a.weights = expert_weights;
    a.out = static_cast<uint16_t *>(hidden_out);
    a.post_weight = static_cast<const uint16_t *>(post_weight);
    a.live = tokens;
    a.top_k = top_k;
    a.hidden = hidden;
    a.routed_scale = routed_scale;
    a.post_eps = post_eps;
    a.has_norm = has_post_norm ? 1 : 0;
    a.status = d->status;
    a.timeout_ns = kWaitLimitNs;
    a.programmatic = g_programmatic.load() != 0;
    a.residual = static_cast<const uint16_t *>(residual);
    a.next_weight = static_cast<const uint16_t *>(next_weight);
    a.normalized = static_cast<uint16_t *>(normalized_out);
    a.next_eps = next_eps;
    a.has_next = has_next_norm ? 1 : 0;
    a.scale_x = scale_x;
    a.scale_residual = scale_residual;
    return from_launch(mf::launch_beam_bulk(a, d->smem_per_sm, d->num_sms, true,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

mf_variant mf_select_finalize_variant(int64_t num_tokens, int32_t hidden, int32_t top_k) {
    if (num_tokens <= 0) return MF_VARIANT_AUTO;
    if (hidden == mf::kTpHidden && top_k == mf::kTpTopK) {
        const DeviceInfo *d = nullptr;
        if (device_info(&d) != MF_OK) d = nullptr;
        return pick_tp(num_tokens, d);
    }
    if (hidden < 256 || hidden > 8192 || hidden % 256 != 0 || top_k < 1 || top_k > 32)
        return MF_VARIANT_AUTO;
    return MF_VARIANT_BULK;
}

const char *mf_finalize_kernel_name(int64_t num_tokens, int32_t hidden, int32_t top_k,
                                    mf_variant variant) {
    if (num_tokens <= 0 || variant < MF_VARIANT_AUTO || variant > MF_VARIANT_CLUSTER) return "";
    if (hidden != mf::kTpHidden || top_k != mf::kTpTopK) {
        if (hidden < 256 || hidden > 8192 || hidden % 256 != 0 || top_k < 1 || top_k > 32) return "";
        if (variant != MF_VARIANT_AUTO && variant != MF_VARIANT_BULK) return "";
        const DeviceInfo *d = nullptr;
        if (device_info(&d) != MF_OK) d = nullptr;
        if (hidden <= 1024)
            return d != nullptr && mf::tp_warp_groups(num_tokens, hidden, top_k, mf::kWeightFP32,
                                                      d->num_sms) > 0
                       ? "tp_warp_bulk_multi_kernel"
                       : "tp_warp_bulk_kernel";
        return d != nullptr && mf::tp_generic_groups(num_tokens, hidden, top_k, mf::kWeightFP32,
                                                     d->smem_per_sm, d->num_sms) > 0
                   ? "tp_generic_bulk_multi_kernel"
                   : "tp_generic_bulk_kernel";
    }
    const DeviceInfo *d = nullptr;
    if (device_info(&d) != MF_OK) d = nullptr;
    if (variant == MF_VARIANT_AUTO) variant = pick_tp(num_tokens, d);
    switch (variant) {
        case MF_VARIANT_CLUSTER: return "tp_cluster_kernel";
        case MF_VARIANT_TOKEN_CTA: return "tp_token_cta_kernel";
        case MF_VARIANT_BULK:
            return d != nullptr && mf::tp_bulk_groups(num_tokens, int64_t{d->bulk_per_sm} * d->num_sms) > 0
                       ? "tp_token_bulk_multi_kernel"
                       : "tp_token_bulk_kernel";
        default: return "";
    }
}

const char *mf_beam_kernel_name(int64_t live_tokens, int32_t top_k, int32_t hidden,
                                mf_variant variant, int residual) {
    if (live_tokens <= 0 || top_k < 1 || top_k > 32 || hidden < 256 || hidden > 8192 ||
        hidden % 256 != 0)
        return "";
    if (variant == MF_VARIANT_AUTO || residual) variant = MF_VARIANT_BULK;
    if (variant == MF_VARIANT_TOKEN_CTA) return "beam_token_cta_kernel";
    if (variant != MF_VARIANT_BULK) return "";
    if (hidden <= 1024) return "beam_warp_bulk_kernel";
    const DeviceInfo *d = nullptr;
    if (device_info(&d) != MF_OK) d = nullptr;
    return d != nullptr && mf::beam_bulk_multi(live_tokens, top_k, hidden, residual != 0,
                                               d->smem_per_sm, d->num_sms)
               ? "beam_token_bulk_multi_kernel"
               : "beam_token_bulk_kernel";
}

mf_variant mf_select_beam_variant(int64_t live_tokens, int32_t top_k, int32_t hidden) {
    (void)top_k;
    (void)hidden;
    return pick_beam(live_tokens);
}

mf_status mf_device_status(int clear) {
    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return MF_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof word) != cudaSuccess) return MF_ERR_CUDA;
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess)
            return MF_ERR_CUDA;
    }
    return (word & mf::kStatusWaitTimeout) ? MF_ERR_DEVICE_TIMEOUT : MF_OK;
}

mf_status mf_selftest_wait_timeout(uint64_t timeout_ns, mf_stream_t stream) {
    const DeviceInfo *d = nullptr;
    mf_status st = device_info(&d);
    if (st != MF_OK) return st;
    if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
    return from_launch(mf::launch_wait_timeout_selftest(d->status, timeout_ns,
                                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
