// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mf {

// The finalize+RMSNorm operation is defined for hidden 4096 and top-k 8
// (flashinfer.comm.tp_moe_finalize_rmsnorm, API page).
constexpr int kTpHidden = 4096;
constexpr int kTpTopK = 8;
constexpr int kTpRowBytes = kTpHidden * 2;

struct TpArgs {
    const uint16_t *gemm2;       // BF16 [rows, ld]
    int64_t rows;
    int64_t ld;                  // row stride in elements
    const void *weights;         // [T, 8] BF16 or FP32
    const int32_t *idx;          // [T, 8]
    const uint16_t *norm_weight; // BF16 [4096]
    uint16_t *out;               // BF16 [T, 4096]
    int64_t num_tokens;
    float eps;
    float gain_center;
    int before;                  // weight_before_norm
    unsigned *status;            // device status word
    uint64_t timeout_ns;         // bound of every device-side wait
};

struct BeamArgs {
    const uint16_t *x;           // BF16 [capacity, K, H]
    const float *weights;        // FP32 [>= live, K]
    uint16_t *out;               // BF16 [live, H]
    const uint16_t *post_weight; // BF16 [H] or nullptr
    int64_t live;
    int top_k;
    int hidden;
    float routed_scale;
    float post_eps;
    int has_norm;
    unsigned *status;
    uint64_t timeout_ns;
};

// Per-device one-time set-up (kernel attributes).  `smem_optin` is the
// device's opt-in shared memory per block, `smem_per_sm` its shared memory
// per multiprocessor.
cudaError_t prepare_tp_kernels(int smem_optin);
cudaError_t prepare_beam_kernels(int smem_per_sm);

cudaError_t launch_tp_token_cta(const TpArgs &a, bool bf16_weights, cudaStream_t s);
cudaError_t launch_tp_cluster(const TpArgs &a, bool bf16_weights, cudaStream_t s);
cudaError_t launch_tp_bulk(const TpArgs &a, bool bf16_weights, cudaStream_t s);

cudaError_t launch_beam_token_cta(const BeamArgs &a, cudaStream_t s);
cudaError_t launch_beam_bulk(const BeamArgs &a, int smem_per_sm, cudaStream_t s);

cudaError_t launch_wait_timeout_selftest(unsigned *status, uint64_t timeout_ns, cudaStream_t s);

}  // namespace mf
