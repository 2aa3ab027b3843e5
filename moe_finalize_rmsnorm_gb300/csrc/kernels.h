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

// How the routing weights are stored: BF16, FP32, or the producer's packed
// int32 routing words (expert_id << 16) | bf16 weight bits, whose low half is
// the weight.
enum WeightKind : int { kWeightBF16 = 0, kWeightFP32 = 1, kWeightPacked = 2 };

struct TpArgs {
    const uint16_t *gemm2;       // BF16 [rows, ld]
    int64_t rows;
    int64_t ld;                  // row stride in elements
    const void *weights;         // [T, K] BF16, FP32 or packed int32
    const int32_t *idx;          // [T, K]
    const uint16_t *norm_weight; // BF16 [H]
    uint16_t *out;               // BF16 [T, H]
    int64_t num_tokens;
    int hidden;                  // H (4096 for the specialised kernels)
    int top_k;                   // K (8 for the specialised kernels)
    float eps;
    float gain_center;
    int before;                  // weight_before_norm
    unsigned *status;            // device status word
    uint64_t timeout_ns;         // bound of every device-side wait
    bool programmatic;           // launch with programmatic dependent launch
};

struct BeamArgs {
    const uint16_t *x;           // BF16 [capacity, K, H]
    const float *weights;        // FP32 [>= live, K]
    uint16_t *out;               // BF16 [live, H] (the hidden output with a residual)
    const uint16_t *post_weight; // BF16 [H] or nullptr
    int64_t live;
    int top_k;
    int hidden;
    float routed_scale;
    float post_eps;
    int has_norm;
    unsigned *status;
    uint64_t timeout_ns;
    bool programmatic;
    // residual step (beam_moe_finalize_norm_residual_norm); unused otherwise
    const uint16_t *residual;    // BF16 [live, H]
    const uint16_t *next_weight; // BF16 [H] or nullptr
    uint16_t *normalized;        // BF16 [live, H] when has_next
    float next_eps;
    int has_next;
    float scale_x;
    float scale_residual;
};

// Per-device one-time set-up (kernel attributes).  `smem_optin` is the
// device's opt-in shared memory per block, `smem_per_sm` its shared memory
// per multiprocessor.
cudaError_t prepare_tp_kernels(int smem_optin, int smem_per_sm);
// CTAs per SM of the staged (bulk; the smaller of its one- and multi-token
// kernels) and register (token_cta) hidden-4096 kernels, from the occupancy
// calculator (after prepare_tp_kernels).
cudaError_t tp_blocks_per_sm(int *bulk, int *token_cta);
cudaError_t prepare_beam_kernels(int smem_per_sm);

// Hidden 4096, top-k 8.
cudaError_t launch_tp_token_cta(const TpArgs &a, int weight_kind, cudaStream_t s);
cudaError_t launch_tp_cluster(const TpArgs &a, int weight_kind, cudaStream_t s);
// `resident_ctas`: CTAs of the staged kernel resident at once on the device
// (CTAs per SM times SMs); it sets how many tokens run in multi-token CTAs.
cudaError_t launch_tp_bulk(const TpArgs &a, int weight_kind, int resident_ctas, cudaStream_t s);
// Multi-token CTAs of the staged hidden-4096 kernel for a launch (0: one token
// per CTA throughout).
int64_t tp_bulk_groups(int64_t num_tokens, int64_t resident_ctas);
// The hidden-4096 finalize's memory traffic without its arithmetic (a
// measurement aid): one staged CTA per token, the output row is the XOR of the
// words read.
cudaError_t launch_tp_data_movement(const TpArgs &a, int weight_kind, cudaStream_t s);
// Any hidden in 256..8192 (multiple of 256) and top-k in 1..32.
cudaError_t launch_tp_generic(const TpArgs &a, int weight_kind, int smem_per_sm, int num_sms,
                              cudaStream_t s);
// Multi-token warps of a warp-per-token launch, hidden 256..1024 (0: one token
// per warp throughout).
int64_t tp_warp_groups(int64_t num_tokens, int hidden, int top_k, int weight_kind, int num_sms);
// Multi-token CTAs of a generic staged launch (0: one token per CTA throughout).
int64_t tp_generic_groups(int64_t num_tokens, int hidden, int top_k, int weight_kind,
                          int smem_per_sm, int num_sms);

cudaError_t launch_beam_token_cta(const BeamArgs &a, cudaStream_t s);
// `residual`: finalize, then the residual-add and next norm of
// beam_moe_finalize_norm_residual_norm.
cudaError_t launch_beam_bulk(const BeamArgs &a, int smem_per_sm, int num_sms, bool residual,
                             cudaStream_t s);
// Whether a staged Beam launch runs the several-tokens-per-CTA kernel.
bool beam_bulk_multi(int64_t live, int top_k, int hidden, bool residual, int smem_per_sm,
                     int num_sms);

cudaError_t launch_wait_timeout_selftest(unsigned *status, uint64_t timeout_ns, cudaStream_t s);

}  // namespace mf
