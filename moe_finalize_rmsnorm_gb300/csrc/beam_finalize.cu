// Beam finalize kernels (sm_103a).
//
// Operation (vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize:
// "reduce only output rows, preserving BF16 casts before scale and RMSNorm"):
//   s[h] = sum_k w[t,k] * x[t,k,h]         FP32 FMA chain, ascending k
//   r    = BF16(s)                          first round
//   v    = BF16(float(r) * routed_scale)    FP32 product, second round
//   norm: out = BF16(v * rsqrt(mean(v^2) + post_eps) * post_weight)
//   else: out = v
// for live tokens t < live_tokens only.
//
// The input is token-major, so a token's K rows are one contiguous block of
// K*H*2 bytes (114,688 B at H = 7168, K = 8) and no index map is involved.
//
//   beam_token_cta_kernel  one CTA per live token, H/8/CPT threads, each owning
//                          CPT 16-byte chunks; slots are loaded in groups of 8
//                          with every load of a group issued before its FMAs.
//   beam_ring_kernel       persistent, one CTA per SM: a producer thread copies
//                          each token's block in units of whole rows (<= 16 KB)
//                          into a shared-memory ring with 1-D bulk copies;
//                          consumer warps reduce, round, scale and normalise.
//
// H ranges over 256..8192 in steps of 256 and K over 1..32, as the wrapper's
// assertions allow.

#include "common.cuh"
#include "kernels.h"

namespace mf {
namespace {

// Round the FP32 sums to BF16, multiply by the scale in FP32, round again.
template <int CPT>
__device__ __forceinline__ void round_scale_round(float (&acc)[CPT][8], float scale) {
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = round_bf16(__fmul_rn(round_bf16(acc[c][j]), scale));
}

template <int CPT>
__device__ __forceinline__ float sum_squares(const float (&v)[CPT][8]) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = __fmaf_rn(v[c][j], v[c][j], ss);
    return ss;
}

// Store v (no norm) or v * rs * post_weight, rounded to BF16.
template <int CPT>
__device__ __forceinline__ void beam_store(const float (&v)[CPT][8], const BeamArgs &a, bool norm,
                                           float rs, uint16_t *out_row, int chunk0, int stride) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int chunk = chunk0 + c * stride;
        float y[8];
        if (norm) {
            float pw[8];
            if (a.post_weight) {
                unpack8(__ldg(reinterpret_cast<const uint4 *>(a.post_weight) + chunk), pw);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) pw[j] = 1.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(__fmul_rn(v[c][j], rs), pw[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = v[c][j];  // already BF16 values: exact
        }
        st_cs_16(out_row + static_cast<int64_t>(chunk) * kChunkElems, pack8_rn(y));
    }
}

__device__ __forceinline__ float inv_rms(float total, int hidden, float eps) {
    return rsqrtf(__fadd_rn(__fdiv_rn(total, static_cast<float>(hidden)), eps));
}

// ---------------------------------------------------------------------------
// one CTA per live token

// Largest block each chunks-per-thread choice can be launched with (see beam_cpt).
template <int CPT>
constexpr int beam_max_threads() { return CPT == 4 ? 256 : (CPT == 2 ? 512 : 1024); }

template <int CPT>
__global__ void __launch_bounds__(beam_max_threads<CPT>()) beam_token_cta_kernel(const BeamArgs a) {
    __shared__ float red[32];
    const int NT = blockDim.x;
    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x;
    const int K = a.top_k, H = a.hidden;
    const uint16_t *xt = a.x + t * K * static_cast<int64_t>(H);
    const float *wt = a.weights + t * K;

    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += 8) {
        const int kn = K - k0 < 8 ? K - k0 : 8;
        uint4 q[8][CPT];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < kn) {
                const uint16_t *row = xt + static_cast<int64_t>(k0 + k) * H;
#pragma unroll
                for (int c = 0; c < CPT; ++c)
                    q[k][c] = ld_nc_na_16(row + (tid + c * NT) * kChunkElems);
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < kn) {
                const float w = __ldg(wt + k0 + k);
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float x[8];
                    unpack8(q[k][c], x);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w, x[j], acc[c][j]);
                }
            }
        }
    }

    round_scale_round<CPT>(acc, a.routed_scale);
    const bool norm = a.has_norm != 0;
    float rs = 1.f;
    if (norm) {
        const float ss = warp_sum(sum_squares<CPT>(acc));
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        const int nw = NT >> 5;
        for (int i = 0; i < nw; ++i) tot += red[i];
        rs = inv_rms(tot, H, a.post_eps);
    }
    beam_store<CPT>(acc, a, norm, rs, a.out + t * H, tid, NT);
}

// ---------------------------------------------------------------------------
// persistent bulk-copy ring

struct BeamRing {
    int slots;
    int rows_per_unit;
    int unit_bytes;
    size_t bytes;
    size_t full, empty, redbar, red;
};

__host__ __device__ inline BeamRing beam_ring_layout(int slots, int rows_per_unit, int hidden) {
    BeamRing L;
    L.slots = slots;
    L.rows_per_unit = rows_per_unit;
    L.unit_bytes = rows_per_unit * hidden * 2;
    size_t off = static_cast<size_t>(slots) * L.unit_bytes;
    L.full = off;   off += sizeof(uint64_t) * slots;
    L.empty = off;  off += sizeof(uint64_t) * slots;
    L.redbar = off; off += sizeof(uint64_t) * 2;
    L.red = off;    off += sizeof(float) * 2 * 32;
    L.bytes = off;
    return L;
}

constexpr int kMaxUnitBytes = 16384;

template <int CPT>
__global__ void __launch_bounds__(beam_max_threads<CPT>() == 1024 ? 1024 : beam_max_threads<CPT>() + 32, 1)
    beam_ring_kernel(const BeamArgs a, const int slots, const int rows_per_unit) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = a.hidden, K = a.top_k;
    const BeamRing L = beam_ring_layout(slots, rows_per_unit, H);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *redbar = reinterpret_cast<uint64_t *>(smem + L.redbar);
    float *red = reinterpret_cast<float *>(smem + L.red);
    const uint32_t ring_base = smem_u32(smem);

    const int NC = blockDim.x - 32;
    const int NCW = NC >> 5;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < slots; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), NCW);
        }
        mbar_init(smem_u32(&redbar[0]), NCW);
        mbar_init(smem_u32(&redbar[1]), NCW);
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t T = a.live;
    const int64_t stride = gridDim.x;
    const int units = K / rows_per_unit;
    const int64_t token_elems = static_cast<int64_t>(K) * H;

    if (tid >= NC) {
        // ------------------------------------------------------ producer
        if (tid != NC) return;
        const uint64_t policy = policy_evict_first();
        uint32_t pos = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < T && ok; t += stride) {
            const uint16_t *src = a.x + t * token_elems;
            for (int u = 0; u < units; ++u) {
                const int s = pos % slots;
                const uint32_t ph = (pos / slots) & 1u;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.timeout_ns)) { ok = false; break; }
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, L.unit_bytes);
                bulk_copy_g2s_hint(ring_base + static_cast<uint32_t>(s) * L.unit_bytes,
                                   src + static_cast<int64_t>(u) * rows_per_unit * H, L.unit_bytes,
                                   fb, policy);
                ++pos;
            }
        }
        if (!ok) {
            atomicOr(a.status, kStatusWaitTimeout);
            const uint32_t first = pos > static_cast<uint32_t>(slots) ? pos - slots : 0u;
            for (uint32_t p = first; p < pos; ++p)
                (void)mbar_wait(smem_u32(&full[p % slots]), (p / slots) & 1u, a.timeout_ns);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31, warp = tid >> 5;
    const bool norm = a.has_norm != 0;
    uint32_t pos = 0, titer = 0;
    int64_t t = blockIdx.x;
    // lane k holds w[t, k]; the next token's weights are fetched one token ahead
    float wnext = (t < T && lane < K) ? __ldg(a.weights + t * K + lane) : 0.f;
    for (; t < T; t += stride, ++titer) {
        const float wl = wnext;
        if (t + stride < T && lane < K) wnext = __ldg(a.weights + (t + stride) * K + lane);

        float acc[CPT][8];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

        for (int u = 0; u < units; ++u) {
            const int s = pos % slots;
            const uint32_t ph = (pos / slots) & 1u;
            if (!mbar_wait(smem_u32(&full[s]), ph, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                return;
            }
            const uint32_t slot = ring_base + static_cast<uint32_t>(s) * L.unit_bytes;
            for (int r = 0; r < rows_per_unit; ++r) {
                const float w = __shfl_sync(0xffffffffu, wl, u * rows_per_unit + r);
                const uint32_t row = slot + static_cast<uint32_t>(r) * H * 2;
                uint4 q[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) q[c] = lds_16(row + (tid + c * NC) * kChunkBytes);
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float x[8];
                    unpack8(q[c], x);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w, x[j], acc[c][j]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            ++pos;
        }

        round_scale_round<CPT>(acc, a.routed_scale);
        float rs = 1.f;
        if (norm) {
            const float ss = warp_sum(sum_squares<CPT>(acc));
            const int b = titer & 1;
            if (lane == 0) {
                red[b * 32 + warp] = ss;
                mbar_arrive(smem_u32(&redbar[b]));
            }
            if (!mbar_wait(smem_u32(&redbar[b]), (titer >> 1) & 1u, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                return;
            }
            float tot = 0.f;
            for (int i = 0; i < NCW; ++i) tot += red[b * 32 + i];
            rs = inv_rms(tot, H, a.post_eps);
        }
        beam_store<CPT>(acc, a, norm, rs, a.out + t * H, tid, NC);
    }
}

// Chunks per thread: the largest of 4, 2, 1 that divides H/256 and leaves at
// least 128 threads (a multiple of 32 either way).
int beam_cpt(int hidden) {
    const int groups = hidden / 256;
    for (int cpt : {4, 2})
        if (groups % cpt == 0 && hidden / 8 / cpt >= 128) return cpt;
    return 1;
}

// Whole rows per ring unit: the largest divisor of K whose rows fit 16 KB.
int beam_rows_per_unit(int top_k, int hidden) {
    for (int r = top_k; r > 1; --r)
        if (top_k % r == 0 && r * hidden * 2 <= kMaxUnitBytes) return r;
    return 1;
}

int beam_slots(int smem_optin, int rows_per_unit, int hidden) {
    int slots = 1;
    while (beam_ring_layout(slots + 1, rows_per_unit, hidden).bytes <=
           static_cast<size_t>(smem_optin))
        ++slots;
    return slots;
}

__global__ void wait_timeout_selftest_kernel(unsigned *status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: phase 0 never completes
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0u, timeout_ns))
        atomicOr(status, kStatusWaitTimeout);
}

}  // namespace

cudaError_t prepare_beam_kernels(int smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(beam_ring_kernel<1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(beam_ring_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_optin);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(beam_ring_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_optin);
    return e;
}

cudaError_t launch_beam_token_cta(const BeamArgs &a, cudaStream_t s) {
    const int cpt = beam_cpt(a.hidden);
    const dim3 grid(static_cast<unsigned>(a.live)), block(a.hidden / 8 / cpt);
    switch (cpt) {
        case 4: beam_token_cta_kernel<4><<<grid, block, 0, s>>>(a); break;
        case 2: beam_token_cta_kernel<2><<<grid, block, 0, s>>>(a); break;
        default: beam_token_cta_kernel<1><<<grid, block, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_beam_ring(const BeamArgs &a, int num_sms, int smem_optin, cudaStream_t s) {
    const int cpt = beam_cpt(a.hidden);
    const int rpu = beam_rows_per_unit(a.top_k, a.hidden);
    const int slots = beam_slots(smem_optin, rpu, a.hidden);
    const size_t bytes = beam_ring_layout(slots, rpu, a.hidden).bytes;
    const int64_t grid = a.live < num_sms ? a.live : num_sms;
    const dim3 block(a.hidden / 8 / cpt + 32);
    switch (cpt) {
        case 4: beam_ring_kernel<4><<<static_cast<unsigned>(grid), block, bytes, s>>>(a, slots, rpu); break;
        case 2: beam_ring_kernel<2><<<static_cast<unsigned>(grid), block, bytes, s>>>(a, slots, rpu); break;
        default: beam_ring_kernel<1><<<static_cast<unsigned>(grid), block, bytes, s>>>(a, slots, rpu); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned *status, uint64_t timeout_ns, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace mf
