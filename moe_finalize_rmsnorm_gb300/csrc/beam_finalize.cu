// Beam finalize kernels (sm_103a).
//
// Operation (vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize: only the
// output rows are reduced, and the BF16 rounds before the scale and before the
// norm are kept):
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
//   beam_token_bulk_kernel one CTA per live token; the token's contiguous block
//                          goes into shared memory by 1-D bulk copies, one per
//                          row, issued by lanes of warp 0 right after the
//                          dependency wait (two CTAs per SM), then every thread
//                          reduces its chunks from shared memory.
//   beam_token_bulk_multi_kernel  hidden 4096..7168: the staged kernel with
//                          several tokens per CTA and a ring of one or two token
//                          slots, the next tokens' rows in flight during the
//                          current token's epilogue (the residual op from five
//                          waves of tokens; plain Beam where two tokens fit a
//                          CTA's buffer or one token per CTA leaves little in
//                          flight).
//   beam_warp_bulk_kernel  hidden 256..1024: the same with one warp per token
//                          (one copy per piece of rows), four tokens per CTA.
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

// post_weight chunks of this thread (BF16 packed), loaded early so the
// epilogue does not wait on them; ones when absent.
template <int CPT>
__device__ __forceinline__ void load_post_weight(const BeamArgs &a, int chunk0, int stride,
                                                 uint4 (&pw)[CPT]) {
#pragma unroll
    for (int c = 0; c < CPT; ++c)
        pw[c] = a.post_weight ? __ldg(reinterpret_cast<const uint4 *>(a.post_weight) + chunk0 +
                                      c * stride)
                              : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
}

// Store v (no norm) or v * rs * post_weight, rounded to BF16.
template <int CPT>
__device__ __forceinline__ void beam_store(const float (&v)[CPT][8], const uint4 (&pwq)[CPT],
                                           bool norm, float rs, uint16_t *out_row, int chunk0,
                                           int stride) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        float y[8];
        if (norm) {
            float pw[8];
            unpack8(pwq[c], pw);
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(__fmul_rn(v[c][j], rs), pw[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = v[c][j];  // already BF16 values: exact
        }
        st_cs_16(out_row + static_cast<int64_t>(chunk0 + c * stride) * kChunkElems, pack8_rn(y));
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
    pdl_wait();

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
    uint4 pwq[CPT];
    load_post_weight<CPT>(a, tid, NT, pwq);
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
    beam_store<CPT>(acc, pwq, norm, rs, a.out + t * H, tid, NT);
}

// Residual step of beam_moe_finalize_norm_residual_norm (residual and
// next_weight chunks are loaded by the caller while the rows are in flight):
// the finalized value
// f = BF16(v * rs * post_weight) (or v), then hidden = BF16(s0 f + s1 residual)
// in FP32 (one product, one FMA), stored; with the next norm, normalized =
// BF16(hidden * rsqrt(mean(hidden^2) + next_eps) * next_weight).  Each thread
// reads the residual chunks it later overwrites (with coherent loads, not the
// read-only path), so hidden may be written into the residual buffer itself.
// WARP: one warp holds the whole token (the RMS is a warp reduction, `red`
// unused); otherwise the CTA does (a shared-memory reduction over NT/32 warps).
template <int CPT, bool WARP = false>
__device__ __forceinline__ void residual_epilogue(float (&v)[CPT][8], const uint4 (&pwq)[CPT],
                                                  const uint4 (&resq)[CPT],
                                                  const uint4 (&nwq)[CPT], const BeamArgs &a,
                                                  bool norm, float rs, int64_t t, int tid, int NT,
                                                  float *red, bool ok) {
    const int H = a.hidden;
    uint16_t *hid_row = a.out + t * H;
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int chunk = tid + c * NT;
        float r[8];
        unpack8(resq[c], r);
        float pw[8];
        unpack8(pwq[c], pw);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float f = norm ? round_bf16(__fmul_rn(__fmul_rn(v[c][j], rs), pw[j])) : v[c][j];
            const float h = round_bf16(__fmaf_rn(a.scale_residual, r[j], __fmul_rn(a.scale_x, f)));
            v[c][j] = h;
            ss = __fmaf_rn(h, h, ss);
        }
        if (ok) st_cs_16(hid_row + static_cast<int64_t>(chunk) * kChunkElems, pack8_rn(v[c]));
    }
    if (!a.has_next) return;
    ss = warp_sum(ss);
    float tot = ss;
    if constexpr (!WARP) {
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        tot = 0.f;
        const int nw = NT >> 5;
        for (int i = 0; i < nw; ++i) tot += red[i];
    }
    const float rn = inv_rms(tot, H, a.next_eps);
    uint16_t *norm_row = a.normalized + t * H;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int chunk = tid + c * NT;
        float g[8];
        unpack8(nwq[c], g);
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(__fmul_rn(v[c][j], rn), g[j]);
        if (ok) st_cs_16(norm_row + static_cast<int64_t>(chunk) * kChunkElems, pack8_rn(y));
    }
}

// ---------------------------------------------------------------------------
// one CTA per live token, the token's rows staged in shared memory

// The token's rows move with one bulk copy per row into a buffer of one piece
// of rows (beam_bulk_rows: all 8 rows, 114,688 B, at H = 7168 and top_k 8),
// each row completing on its own mbarrier; lane r of warp 0 issues row r of the
// first piece.  Data in flight holds no registers, and two CTAs per SM keep two
// tokens' blocks in flight while one of them reduces.  Rows beyond one piece
// are copied piece by piece into the same buffer by thread 0.
// PER_ROW: one mbarrier per buffered row (rows of 4 KB and more); otherwise
// one copy and one mbarrier per piece (small rows).
template <int CPT, bool RESID, bool PER_ROW>
__global__ void __launch_bounds__(beam_max_threads<CPT>(), CPT == 2 ? 2 : 1)
    beam_token_bulk_kernel(const BeamArgs a, const int rows_per_piece) {
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[PER_ROW ? 32 : 1];
    __shared__ float red[32];
    __shared__ float red2[32];
    __shared__ float wsm[32];
    const int NT = blockDim.x;
    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x;
    const int K = a.top_k, H = a.hidden;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2;
    const uint32_t base = smem_u32(rows_smem);
    const uint16_t *xt = a.x + t * K * static_cast<int64_t>(H);

    // Copy k0..k0+n-1 of the token's rows into the buffer (thread 0: the pieces
    // after the first, and the first one for small rows).  One mbarrier per
    // buffered row: the reduction starts on a row as soon as it lands.
    auto issue_piece = [&](int k0, int n) {
        const uint64_t policy = policy_evict_first();
        if (PER_ROW) {
            for (int r = 0; r < n; ++r) {
                const uint32_t b = smem_u32(&bars[r]);
                mbar_arrive_expect_tx(b, row_bytes);
                bulk_copy_g2s_hint(base + r * row_bytes, xt + static_cast<int64_t>(k0 + r) * H,
                                   row_bytes, b, policy);
            }
        } else {  // the piece's rows are contiguous: one copy
            const uint32_t b = smem_u32(&bars[0]);
            mbar_arrive_expect_tx(b, n * row_bytes);
            bulk_copy_g2s_hint(base, xt + static_cast<int64_t>(k0) * H, n * row_bytes, b, policy);
        }
    };
    // The rows' addresses depend on nothing the kernel reads, so the first
    // piece goes in flight at once: with per-row barriers lane r of warp 0
    // initialises and arms row r's mbarrier and copies row r (all in parallel),
    // otherwise thread 0 copies the piece.
    const int n0 = K < rows_per_piece ? K : rows_per_piece;
    if (PER_ROW) {
        if (tid < rows_per_piece) {
            mbar_init(smem_u32(&bars[tid]), 1);
            fence_mbar_init();
        }
        pdl_wait();
        if (tid < n0) {
            const uint32_t b = smem_u32(&bars[tid]);
            mbar_arrive_expect_tx(b, row_bytes);
            bulk_copy_g2s_hint(base + tid * row_bytes, xt + static_cast<int64_t>(tid) * H, row_bytes, b,
                               policy_evict_first());
        }
    } else {
        if (tid == 0) {
            mbar_init(smem_u32(&bars[0]), 1);
            fence_mbar_init();
        }
        pdl_wait();
        if (tid == 0) issue_piece(0, n0);
    }
    if (tid < K) wsm[tid] = __ldg(a.weights + t * K + tid);
    uint4 pwq[CPT];  // post_weight, fetched while the rows are in flight
    load_post_weight<CPT>(a, tid, NT, pwq);
    uint4 resq[CPT], nwq[CPT];  // residual step: residual and next_weight chunks, same
    if constexpr (RESID) {
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int chunk = tid + c * NT;
            resq[c] = ld_na_16(a.residual + t * H + static_cast<int64_t>(chunk) * kChunkElems);
            nwq[c] = a.next_weight
                         ? __ldg(reinterpret_cast<const uint4 *>(a.next_weight) + chunk)
                         : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        }
    }
    __syncthreads();

    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

    bool ok = true;
    uint32_t phase = 0;
    for (int k0 = 0; k0 < K; k0 += rows_per_piece, phase ^= 1u) {
        const int n = K - k0 < rows_per_piece ? K - k0 : rows_per_piece;
        if (tid == 0 && k0 > 0) {
            fence_proxy_async_smem();  // earlier reads of the buffer come first
            issue_piece(k0, n);
        }
        for (int r = 0; r < n; ++r) {
            if (PER_ROW || r == 0) {
                const uint32_t b = smem_u32(&bars[PER_ROW ? r : 0]);
                if (!mbar_wait(b, phase, a.timeout_ns)) {
                    atomicOr(a.status, kStatusWaitTimeout);
                    ok = false;
                    (void)mbar_wait(b, phase, a.timeout_ns);  // bounded: the copy may land, or not, before exit
                }
            }
            const float w = wsm[k0 + r];
            const uint32_t row = base + static_cast<uint32_t>(r) * row_bytes;
            uint4 q[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) q[c] = lds_16(row + (tid + c * NT) * kChunkBytes);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float x[8];
                unpack8(q[c], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w, x[j], acc[c][j]);
            }
        }
        if (k0 + rows_per_piece < K) __syncthreads();  // the next piece reuses the buffer
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
    if constexpr (RESID) {
        residual_epilogue<CPT>(acc, pwq, resq, nwq, a, norm, rs, t, tid, NT, red2, ok);
    } else {
        if (ok) beam_store<CPT>(acc, pwq, norm, rs, a.out + t * H, tid, NT);
    }
}

// The staged kernel with several tokens per CTA and a ring of token slots, for
// two chunks per thread (hidden 2048..7168, up to 448 threads) and a token
// whose rows fit one slot with a barrier per row.  CTA b < groups takes n
// consecutive live tokens, the CTAs after it u each (the last one fewer).  A
// CTA first puts up to `slots` tokens in flight, one row copy per lane of warp
// 0; once every thread has read a token's rows, those lanes copy the token
// `slots` ahead into the same slot, before the current token's epilogue, so the
// serial end of each token (its RMS reductions, the residual step, the stores)
// overlaps row traffic.  The weights of a slot's token are stored by the lanes
// that copy its rows, before they arm the row barriers (whose release orders
// them before every reader's acquire).  Each token's arithmetic is that of
// beam_token_bulk_kernel: the same bits.
constexpr int kBeamTokensPerCta = 3;  // n = 3 x slots: as the finalize's multi-token kernels
constexpr int kBeamSingleWaves = 2;   // waves of u-token CTAs at the end
constexpr int kBeamMultiCPT = 2;
// At most 448 threads (hidden 7168) so that two CTAs keep 72 registers per
// thread: 512 threads would leave 64, fewer than the residual form needs.
constexpr int kBeamMultiMaxThreads = 448;
constexpr int kBeamMultiBars = 32;  // slots x top_k row barriers

struct BeamMultiLayout {
    int64_t groups;  // CTAs b < groups take n tokens, the later ones u
    int n;
    int u;
    int slots;       // tokens whose rows the buffer holds at once
    int compact;     // plain Beam built for three CTAs per SM (fewer registers)
};

// MINB 3 (plain Beam only): held to the registers of three 448-thread CTAs
// (40, with a 16-byte spill), so that at hidden 4096..6656 it runs as many
// CTAs per SM as the one-token kernel, which the 2-block build (59 registers)
// does not.
template <bool RESID, int MINB = 2>
__global__ void __launch_bounds__(kBeamMultiMaxThreads, MINB)
    beam_token_bulk_multi_kernel(const BeamArgs a, const BeamMultiLayout lay) {
    constexpr int CPT = kBeamMultiCPT;
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[kBeamMultiBars];
    __shared__ float red[2][32];
    __shared__ float red2[2][32];
    __shared__ float wsm[kBeamMultiBars];  // slot s, row r at s * K + r
    const int NT = blockDim.x;
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    int64_t t0;
    int cnt;
    if (b < lay.groups) {
        t0 = lay.n * b;
        cnt = lay.n;
    } else {
        t0 = int64_t{lay.n} * lay.groups + int64_t{lay.u} * (b - lay.groups);
        const int64_t left = a.live - t0;
        cnt = left < lay.u ? static_cast<int>(left) : lay.u;
    }
    const int K = a.top_k, H = a.hidden, S = lay.slots;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2;
    const uint32_t token_bytes = row_bytes * static_cast<uint32_t>(K);
    const uint32_t base = smem_u32(rows_smem);

    // lane s * K + r of warp 0 copies row r of the token in slot s
    auto issue = [&](int slot, int r, int64_t tok) {
        const uint32_t bb = smem_u32(&bars[slot * K + r]);
        mbar_arrive_expect_tx(bb, row_bytes);
        bulk_copy_g2s_hint(base + slot * token_bytes + r * row_bytes,
                           a.x + (tok * K + r) * static_cast<int64_t>(H), row_bytes, bb,
                           policy_evict_first());
    };
    const int first = cnt < S ? cnt : S;
    if (tid < S * K) {
        mbar_init(smem_u32(&bars[tid]), 1);
        fence_mbar_init();
    }
    pdl_wait();
    if (tid < first * K) {
        const int slot = tid / K, r = tid - slot * K;
        issue(slot, r, t0 + slot);
        wsm[tid] = __ldg(a.weights + (t0 + slot) * K + r);
    }
    uint4 pwq_cta[CPT];  // plain Beam: post_weight held across the tokens
    if (!RESID) load_post_weight<CPT>(a, tid, NT, pwq_cta);
    __syncthreads();  // barriers initialised, first weights stored

    const bool norm = a.has_norm != 0;
    int slot = 0;
    uint32_t phase = 0;
    for (int j = 0; j < cnt; ++j) {
        const int64_t t = t0 + j;
        uint4 resq[CPT];
        if (RESID) {  // this token's residual chunks, while its rows land
#pragma unroll
            for (int c = 0; c < CPT; ++c)
                resq[c] = ld_na_16(a.residual + t * H + static_cast<int64_t>(tid + c * NT) * kChunkElems);
        }
        const bool refill = j + S < cnt;
        const float wnext = (refill && tid < K) ? __ldg(a.weights + (t + S) * K + tid) : 0.f;
        float acc[CPT][8];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
        bool ok = true;
        for (int r = 0; r < K; ++r) {
            const uint32_t bb = smem_u32(&bars[slot * K + r]);
            if (!mbar_wait(bb, phase, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                ok = false;
                (void)mbar_wait(bb, phase, a.timeout_ns);  // bounded: the copy may land, or not, before exit
            }
            const float w = wsm[slot * K + r];
            const uint32_t row = base + slot * token_bytes + static_cast<uint32_t>(r) * row_bytes;
            uint4 q[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) q[c] = lds_16(row + (tid + c * NT) * kChunkBytes);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float x[8];
                unpack8(q[c], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[c][e] = __fmaf_rn(w, x[e], acc[c][e]);
            }
        }
        bool more = true;
        if (refill) {
            // every thread has read this slot and none gave up waiting: the
            // token `slots` ahead goes in flight into it before this epilogue
            more = !__syncthreads_or(!ok);
            if (more && tid < K) {
                wsm[slot * K + tid] = wnext;
                fence_proxy_async_smem();  // the reads above come before the copy
                issue(slot, tid, t + S);
            }
        }
        uint4 pwq[CPT], nwq[CPT];
        if (RESID) {
            // post_weight and next_weight (the same for every token, so mostly
            // cache hits) are requested here, not across the row loop, to
            // spare registers
            load_post_weight<CPT>(a, tid, NT, pwq);
#pragma unroll
            for (int c = 0; c < CPT; ++c)
                nwq[c] = a.next_weight
                             ? __ldg(reinterpret_cast<const uint4 *>(a.next_weight) + tid + c * NT)
                             : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        } else {
#pragma unroll
            for (int c = 0; c < CPT; ++c) pwq[c] = pwq_cta[c];
        }
        round_scale_round<CPT>(acc, a.routed_scale);
        float rs = 1.f;
        if (norm) {
            float *rd = red[j & 1];  // alternate: a slow warp may still read the last one
            const float ss = warp_sum(sum_squares<CPT>(acc));
            if ((tid & 31) == 0) rd[tid >> 5] = ss;
            __syncthreads();
            float tot = 0.f;
            const int nw = NT >> 5;
            for (int i = 0; i < nw; ++i) tot += rd[i];
            rs = inv_rms(tot, H, a.post_eps);
        }
        if (RESID) {
            residual_epilogue<CPT>(acc, pwq, resq, nwq, a, norm, rs, t, tid, NT, red2[j & 1], ok);
        } else if (ok) {
            beam_store<CPT>(acc, pwq, norm, rs, a.out + t * H, tid, NT);
        }
        if (!more) break;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
}

// ---------------------------------------------------------------------------
// small hidden (256..1024): one warp per live token, four tokens per CTA

// As beam_token_bulk_kernel, with one warp per token: lane 0 copies the
// token's contiguous rows into the warp's slice of shared memory (at most
// 16 KB, one copy and one mbarrier per piece), each lane owns CPW 16-byte
// chunks (hidden = 256 CPW), and both RMS reductions are warp reductions.
constexpr int kBeamWarpTokens = 4;
constexpr int kBeamWarpSlice = 16384;

template <int CPW, bool RESID>
__global__ void __launch_bounds__(32 * kBeamWarpTokens)
    beam_warp_bulk_kernel(const BeamArgs a, const int rows_per_piece) {
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[kBeamWarpTokens];
    constexpr int H = 256 * CPW;
    constexpr uint32_t row_bytes = H * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kBeamWarpTokens + warp;
    if (t >= a.live) return;
    const int K = a.top_k;
    const uint32_t base = smem_u32(rows_smem) + warp * rows_per_piece * row_bytes;
    const uint32_t bar = smem_u32(&bars[warp]);
    const uint16_t *xt = a.x + t * K * static_cast<int64_t>(H);

    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    pdl_wait();
    const float wl = lane < K ? __ldg(a.weights + t * K + lane) : 0.f;
    uint4 pwq[CPW];
    load_post_weight<CPW>(a, lane, 32, pwq);
    uint4 resq[CPW], nwq[CPW];
    if constexpr (RESID) {
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            const int chunk = lane + c * 32;
            resq[c] = ld_na_16(a.residual + t * H + static_cast<int64_t>(chunk) * kChunkElems);
            nwq[c] = a.next_weight
                         ? __ldg(reinterpret_cast<const uint4 *>(a.next_weight) + chunk)
                         : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        }
    }
    __syncwarp();

    float acc[CPW][8];
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;
    bool ok = true;
    uint32_t phase = 0;
    for (int k0 = 0; k0 < K; k0 += rows_per_piece, phase ^= 1u) {
        const int n = K - k0 < rows_per_piece ? K - k0 : rows_per_piece;
        if (lane == 0) {
            if (k0 > 0) fence_proxy_async_smem();  // earlier reads of the slice come first
            mbar_arrive_expect_tx(bar, n * row_bytes);
            bulk_copy_g2s_hint(base, xt + static_cast<int64_t>(k0) * H, n * row_bytes, bar,
                               policy_evict_first());
        }
        if (!mbar_wait(bar, phase, a.timeout_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            ok = false;
            (void)mbar_wait(bar, phase, a.timeout_ns);  // bounded: the copy may land, or not, before exit
        }
        for (int r = 0; r < n; ++r) {
            const float w = __shfl_sync(0xffffffffu, wl, k0 + r);
            const uint32_t row = base + r * row_bytes;
            uint4 q[CPW];
#pragma unroll
            for (int c = 0; c < CPW; ++c) q[c] = lds_16(row + (lane + c * 32) * kChunkBytes);
#pragma unroll
            for (int c = 0; c < CPW; ++c) {
                float x[8];
                unpack8(q[c], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w, x[j], acc[c][j]);
            }
        }
        __syncwarp();  // the next piece reuses the slice
    }

    round_scale_round<CPW>(acc, a.routed_scale);
    const bool norm = a.has_norm != 0;
    float rs = 1.f;
    if (norm) rs = inv_rms(warp_sum(sum_squares<CPW>(acc)), H, a.post_eps);
    if constexpr (RESID) {
        residual_epilogue<CPW, true>(acc, pwq, resq, nwq, a, norm, rs, t, lane, 32, nullptr, ok);
    } else {
        if (ok) beam_store<CPW>(acc, pwq, norm, rs, a.out + t * H, lane, 32);
    }
}

// Chunks per thread of the register kernel: the largest of 4, 2, 1 that
// divides H/256 and leaves at least 128 threads (a multiple of 32 either way).
int beam_cpt(int hidden) {
    const int groups = hidden / 256;
    for (int cpt : {4, 2})
        if (groups % cpt == 0 && hidden / 8 / cpt >= 128) return cpt;
    return 1;
}

// Chunks per thread of the staged kernel: 2 when that leaves at least 128
// threads (hidden 2048 and up, an even number of 256-column groups), else 1
// (at 2560 and 3584 two measured 3-4 % faster, elsewhere the same).
int beam_bulk_cpt(int hidden) {
    return ((hidden / 256) % 2 == 0 && hidden / 16 >= 128) ? 2 : 1;
}

// Shared memory one staged CTA may use so that two fit on an SM (each CTA
// also takes 1 KB reserved by the system and up to 1 KB of static shared
// memory: barriers, reduction and weight arrays).
int beam_bulk_budget(int smem_per_sm) { return smem_per_sm / 2 - 1024 - 1024; }

// Rows per piece: at least 8 (a whole token at top_k <= 8), otherwise pieces
// sized so that eight CTAs fit an SM, never more than half an SM's shared
// memory (2048 x 32: 1.05 of the copy peak against 0.80 with pieces of half an
// SM; 1280 x 32 1.03 against 0.84; the 8-slot sizes do not change).
int beam_bulk_rows(int smem_per_sm, int top_k, int hidden) {
    int rows = (smem_per_sm / 8 - 2048) / (hidden * 2);
    if (rows < 8) rows = 8;
    const int half = beam_bulk_budget(smem_per_sm) / (hidden * 2);
    if (rows > half) rows = half;
    return rows < 1 ? 1 : (rows > top_k ? top_k : rows);
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

cudaError_t prepare_beam_kernels(int smem_per_sm) {
    const int budget = beam_bulk_budget(smem_per_sm);
    const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaSuccess;
    const int warp_smem = kBeamWarpSlice * kBeamWarpTokens;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<1, false>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<2, false>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<3, false>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<4, false>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<1, true>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<2, true>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<3, true>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_warp_bulk_kernel<4, true>, attr, warp_smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<1, false, false>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<1, true, false>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<1, false, true>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<1, true, true>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<2, false, true>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_kernel<2, true, true>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_multi_kernel<false>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_multi_kernel<false, 3>, attr, budget);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(beam_token_bulk_multi_kernel<true>, attr, budget);
    return e;
}

cudaError_t launch_beam_token_cta(const BeamArgs &a, cudaStream_t s) {
    const int cpt = beam_cpt(a.hidden);
    const dim3 grid(static_cast<unsigned>(a.live)), block(a.hidden / 8 / cpt);
    const bool p = a.programmatic;
    switch (cpt) {
        case 4: return launch_ex(beam_token_cta_kernel<4>, grid, block, 0, s, 1, p, a);
        case 2: return launch_ex(beam_token_cta_kernel<2>, grid, block, 0, s, 1, p, a);
        default: return launch_ex(beam_token_cta_kernel<1>, grid, block, 0, s, 1, p, a);
    }
}

template <int CPW>
static cudaError_t launch_beam_warp(const BeamArgs &a, bool residual, cudaStream_t s) {
    const int fit = kBeamWarpSlice / (a.hidden * 2);
    const int rows = fit < a.top_k ? fit : a.top_k;
    const dim3 grid(static_cast<unsigned>((a.live + kBeamWarpTokens - 1) / kBeamWarpTokens));
    const dim3 block(32 * kBeamWarpTokens);
    const size_t bytes = static_cast<size_t>(rows) * a.hidden * 2 * kBeamWarpTokens;
    if (residual)
        return launch_ex(beam_warp_bulk_kernel<CPW, true>, grid, block, bytes, s, 1, a.programmatic, a, rows);
    return launch_ex(beam_warp_bulk_kernel<CPW, false>, grid, block, bytes, s, 1, a.programmatic, a, rows);
}

template <bool RESID>
static int beam_multi_per_sm(int threads, size_t bytes) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, beam_token_bulk_multi_kernel<RESID>,
                                                      threads, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

static int beam_compact_per_sm(int threads, size_t bytes) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, beam_token_bulk_multi_kernel<false, 3>,
                                                      threads, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <bool RESID>
static int beam_one_per_sm(int threads, size_t bytes) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, beam_token_bulk_kernel<kBeamMultiCPT, RESID, true>, threads, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Layout of a launch of the several-tokens kernel (slots 0: one token per CTA
// instead).  It runs at the one-token kernel's CTAs per SM, never fewer: where
// its extra registers would cost a CTA per SM (hidden 4096 / 5120 at small
// top_k) the concurrency of more CTAs measured faster.  Plain Beam may then use
// the build held to three CTAs' registers, with two token slots, where one
// token per CTA leaves under 80 KB in flight per SM (4096 x 1, 4608 x 1 / 2,
// 5632 x 1 / 2, 6144 x 2, 6656 x 2: 3-20 % faster); with more in flight its
// spill and fewer registers cost more than the slots gain (4096 x 2: -2 %,
// 6144 x 3: -7 %).  The residual op holds
// one token per slot ring (more measured slower: its long epilogue, not the
// bytes in flight, sets the pace); plain Beam holds two when two fit (at hidden
// 7168 and top_k 1..4: 10-18 % faster than one token per CTA; four or eight
// slots were slower than two), or one where one token per CTA leaves less than
// 192 KB in flight per SM (hidden 5120 / 5632 at top_k 8: 2-4 % faster; with
// more in flight the same or slower).
static BeamMultiLayout beam_multi_layout(int64_t live, int top_k, int hidden, bool residual,
                                         int smem_per_sm, int num_sms) {
    BeamMultiLayout lay = {0, 0, 0, 0, 0};
    const int threads = hidden / 8 / kBeamMultiCPT;
    // hidden 2048..3584 (more CTAs per SM) measured the same or 0.7-1.5 % slower
    if (hidden < 4096 || beam_bulk_cpt(hidden) != kBeamMultiCPT || threads > kBeamMultiMaxThreads ||
        num_sms <= 0 || live <= 0 || beam_bulk_rows(smem_per_sm, top_k, hidden) < top_k)
        return lay;
    const int64_t token_bytes = int64_t{top_k} * hidden * 2;
    const int occ_one =
        residual ? beam_one_per_sm<true>(threads, static_cast<size_t>(token_bytes))
                 : beam_one_per_sm<false>(threads, static_cast<size_t>(token_bytes));
    const int occ_multi =
        residual ? beam_multi_per_sm<true>(threads, 0) : beam_multi_per_sm<false>(threads, 0);
    int compact = 0;
    if (occ_one <= 0) return lay;
    if (occ_multi < occ_one) {
        if (residual || beam_compact_per_sm(threads, 0) < occ_one) return lay;
        compact = 1;
    }
    int slots = static_cast<int>((smem_per_sm / occ_one - 2048) / token_bytes);
    const int cap = residual ? 1 : 2;
    if (slots > cap) slots = cap;
    if (slots > kBeamMultiBars / top_k) slots = kBeamMultiBars / top_k;
    if (slots < 1) return lay;
    if (!residual && slots < 2 && (compact || occ_one * token_bytes >= 192 * 1024)) return lay;
    if (compact && occ_one * token_bytes >= 80 * 1024) return lay;
    const size_t sbytes = static_cast<size_t>(slots * token_bytes);
    const int per_sm = residual ? beam_multi_per_sm<true>(threads, sbytes)
                       : compact ? beam_compact_per_sm(threads, sbytes)
                                 : beam_multi_per_sm<false>(threads, sbytes);
    const int64_t resident = int64_t{per_sm} * num_sms;
    if (resident <= 0) return lay;
    int64_t u = live / (4 * resident);  // later CTAs small enough for about four waves
    if (u > slots) u = slots;
    if (u < 1) u = 1;
    const int64_t n = int64_t{kBeamTokensPerCta} * slots, singles = kBeamSingleWaves * u * resident;
    int64_t groups = 0;
    if (live >= singles + n * resident) {
        groups = (live - singles) / n;
        const int64_t r = groups % resident;  // drop a partial wave that would outlast the rest
        if (r != 0 && n * (resident - r) > singles) groups -= r;
    }
    if (groups == 0 && u == 1) return lay;  // one token per CTA throughout
    lay.groups = groups;
    lay.n = static_cast<int>(n);
    lay.u = static_cast<int>(u);
    lay.slots = slots;
    lay.compact = compact;
    return lay;
}

bool beam_bulk_multi(int64_t live, int top_k, int hidden, bool residual, int smem_per_sm,
                     int num_sms) {
    return beam_multi_layout(live, top_k, hidden, residual, smem_per_sm, num_sms).slots > 0;
}

cudaError_t launch_beam_bulk(const BeamArgs &a, int smem_per_sm, int num_sms, bool residual,
                             cudaStream_t s) {
    switch (a.hidden) {  // hidden 256..1024: one warp per token
        case 256: return launch_beam_warp<1>(a, residual, s);
        case 512: return launch_beam_warp<2>(a, residual, s);
        case 768: return launch_beam_warp<3>(a, residual, s);
        case 1024: return launch_beam_warp<4>(a, residual, s);
        default: break;
    }
    const int cpt = beam_bulk_cpt(a.hidden);
    const int rows = beam_bulk_rows(smem_per_sm, a.top_k, a.hidden);
    const size_t bytes = static_cast<size_t>(rows) * a.hidden * 2;
    const dim3 grid(static_cast<unsigned>(a.live)), block(a.hidden / 8 / cpt);
    const bool p = a.programmatic;
    const BeamMultiLayout lay = beam_multi_layout(a.live, a.top_k, a.hidden, residual, smem_per_sm, num_sms);
    if (lay.slots > 0) {
        const int64_t ctas = lay.groups + (a.live - int64_t{lay.n} * lay.groups + lay.u - 1) / lay.u;
        const size_t mbytes = static_cast<size_t>(lay.slots) * a.top_k * a.hidden * 2;
        if (residual)
            return launch_ex(beam_token_bulk_multi_kernel<true>, dim3(static_cast<unsigned>(ctas)), block, mbytes, s, 1, p, a, lay);
        if (lay.compact)
            return launch_ex(beam_token_bulk_multi_kernel<false, 3>, dim3(static_cast<unsigned>(ctas)), block, mbytes, s, 1, p, a, lay);
        return launch_ex(beam_token_bulk_multi_kernel<false>, dim3(static_cast<unsigned>(ctas)), block, mbytes, s, 1, p, a, lay);
    }
    // CPT 2 implies hidden >= 2048 (rows of 4 KB and more): per-row barriers
    if (cpt == 2) {
        if (residual) return launch_ex(beam_token_bulk_kernel<2, true, true>, grid, block, bytes, s, 1, p, a, rows);
        return launch_ex(beam_token_bulk_kernel<2, false, true>, grid, block, bytes, s, 1, p, a, rows);
    }
    if (a.hidden >= 2048) {
        if (residual) return launch_ex(beam_token_bulk_kernel<1, true, true>, grid, block, bytes, s, 1, p, a, rows);
        return launch_ex(beam_token_bulk_kernel<1, false, true>, grid, block, bytes, s, 1, p, a, rows);
    }
    if (residual) return launch_ex(beam_token_bulk_kernel<1, true, false>, grid, block, bytes, s, 1, p, a, rows);
    return launch_ex(beam_token_bulk_kernel<1, false, false>, grid, block, bytes, s, 1, p, a, rows);
}

cudaError_t launch_wait_timeout_selftest(unsigned *status, uint64_t timeout_ns, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace mf
