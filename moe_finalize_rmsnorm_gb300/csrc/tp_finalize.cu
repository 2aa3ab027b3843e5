// Finalize + RMSNorm kernels (sm_103a): specialised kernels for hidden 4096,
// top-k 8, and a generic kernel for hidden 256..8192 (multiple of 256) and
// top-k 1..32.
//
// Operation (flashinfer.comm.tp_moe_finalize_rmsnorm, API page):
//   acc[h] = sum over valid slots k (0 <= idx[t,k] < rows), ascending k,
//            of w[t,k] * gemm2[idx[t,k], h]                  FP32 FMA chain
//   g[h]   = float(norm_weight[h]) + gain_center             FP32 add
//   before: v = acc * g; y = v * rsqrt(mean(v^2) + eps)
//   after:  y = acc * rsqrt(mean(acc^2) + eps) * g
//   out    = BF16(y), round to nearest even
//
// The path is a gather-reduce bound by HBM bandwidth: 64 KB of gathered rows
// and 8 KB of output per token.  Three kernels cover the size range:
//
//   tp_token_cta_kernel  one CTA per token; each thread owns CPT 16-byte
//                        column chunks and issues all 8 slot loads for them
//                        before the first FMA, so 8*CPT loads are in flight
//                        per thread.  Sum of squares: warp shuffles + shared
//                        memory.
//   tp_cluster_kernel    decode sizes: a cluster of C CTAs per token, each
//                        CTA owning 4096/C columns; the partial sums of
//                        squares are exchanged through distributed shared
//                        memory, so a token's 64 KB gather spreads over C SMs.
//   tp_token_bulk_kernel one CTA per token; thread 0 stages the token's valid
//                        rows in shared memory with 1-D bulk copies
//                        (cp.async.bulk), one mbarrier per row, so no
//                        registers are held by data in flight and three
//                        CTAs (192 KB of rows) fit per SM.
//   tp_generic_bulk_kernel  any (hidden, top-k) in range: the staged design
//                        with runtime sizes; the valid rows are copied in
//                        pieces of at least 8 rows (at most half an SM's
//                        shared memory), the first piece's rows each by the
//                        lane of its slot.
//   tp_warp_bulk_kernel  hidden 256..1024: the staged design with one warp per
//                        token and two tokens per CTA (small tokens would
//                        otherwise make the grid CTA-launch bound); each
//                        valid slot's lane copies its own row.
//   *_multi_kernel       the three staged kernels above with three tokens in
//                        each of the first CTAs (warps) of a launch of five
//                        waves and more: the next token's route is loaded
//                        while the current rows land, and its rows go in
//                        flight before the current token's norm and stores.
//                        The generic one holds two tokens at once (six per
//                        CTA) when tokens are small (top_k 1..3 at large
//                        hidden), where one token per CTA leaves little in
//                        flight.
//   tp_data_movement_kernel  not part of the operation: the hidden-4096
//                        finalize's memory traffic with no arithmetic, a
//                        measuring stick for the kernels above.
//
// Routing weights may be BF16, FP32 or the producer's packed int32 routing
// words (expert_id << 16) | bf16 weight bits (trtllm_fp8_per_tensor_scale_
// routed_moe, topk_ids parameter), whose low half is the weight.
//
// Every wait on an mbarrier is bounded (TpArgs::timeout_ns); a wait that gives
// up ORs kStatusWaitTimeout into the device status word, waits once more (also
// bounded) for the copies it issued, and the kernel returns without storing.
// If that second wait gives up too, a copy may still be writing into shared
// memory after the CTA has left, so after a timeout the outputs of the call and
// of later kernels on the context are unspecified.

#include "common.cuh"
#include "kernels.h"

namespace mf {
namespace {

constexpr int kChunksPerRow = kTpHidden / kChunkElems;  // 512

// Load the 8 route entries of token t (same address across the block: the
// loads are broadcasts).
template <int WK>
__device__ __forceinline__ void load_route(const TpArgs &a, int64_t t, int (&idx)[8],
                                           float (&w)[8]) {
    const int4 *ip = reinterpret_cast<const int4 *>(a.idx + t * kTpTopK);
    const int4 i0 = __ldg(ip), i1 = __ldg(ip + 1);
    idx[0] = i0.x; idx[1] = i0.y; idx[2] = i0.z; idx[3] = i0.w;
    idx[4] = i1.x; idx[5] = i1.y; idx[6] = i1.z; idx[7] = i1.w;
    if constexpr (WK == kWeightBF16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(
            static_cast<const uint16_t *>(a.weights) + t * kTpTopK));
        unpack8(q, w);
    } else if constexpr (WK == kWeightPacked) {
        const uint4 *pp = reinterpret_cast<const uint4 *>(
            static_cast<const int32_t *>(a.weights) + t * kTpTopK);
        const uint4 p0 = __ldg(pp), p1 = __ldg(pp + 1);
        w[0] = bf16_lo(p0.x); w[1] = bf16_lo(p0.y); w[2] = bf16_lo(p0.z); w[3] = bf16_lo(p0.w);
        w[4] = bf16_lo(p1.x); w[5] = bf16_lo(p1.y); w[6] = bf16_lo(p1.z); w[7] = bf16_lo(p1.w);
    } else {
        const float4 *wp = reinterpret_cast<const float4 *>(
            static_cast<const float *>(a.weights) + t * kTpTopK);
        const float4 w0 = __ldg(wp), w1 = __ldg(wp + 1);
        w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
        w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
    }
}

__device__ __forceinline__ bool slot_valid(int i, int64_t rows) {
    return i >= 0 && static_cast<int64_t>(i) < rows;
}

// g = float(norm_weight) + gain_center for one 16-byte chunk.
__device__ __forceinline__ void load_gain(const TpArgs &a, int chunk, float (&g)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(a.norm_weight) + chunk);
    unpack8(q, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = __fadd_rn(g[j], a.gain_center);
}

// Before-norm: acc <- acc * g.  Returns this thread's sum of squares of the
// values the RMS is taken over.
template <int CPT>
__device__ __forceinline__ float prenorm(float (&acc)[CPT][8], const float (&g)[CPT][8],
                                         bool before) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (before) acc[c][j] = __fmul_rn(acc[c][j], g[c][j]);
            ss = __fmaf_rn(acc[c][j], acc[c][j], ss);
        }
    return ss;
}

// y = v * r (before) or acc * r * g (after), rounded to BF16 and stored.
template <int CPT, int STRIDE>
__device__ __forceinline__ void scale_store(const float (&acc)[CPT][8], const float (&g)[CPT][8],
                                            bool before, float r, uint16_t *out_row, int chunk0) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float s = __fmul_rn(acc[c][j], r);
            y[j] = before ? s : __fmul_rn(s, g[c][j]);
        }
        st_cs_16(out_row + static_cast<int64_t>(chunk0 + c * STRIDE) * kChunkElems, pack8_rn(y));
    }
}

// ---------------------------------------------------------------------------
// one CTA per token

template <int CPT, int WK>
__global__ void __launch_bounds__(kChunksPerRow / CPT)
    tp_token_cta_kernel(const TpArgs a) {
    constexpr int NT = kChunksPerRow / CPT;
    constexpr int NW = NT / 32;
    __shared__ float red[NW];

    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;

    pdl_wait();
    int idx[8];
    float w[8];
    load_route<WK>(a, t, idx, w);

    // issue every gather before the first use
    uint4 q[8][CPT];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool ok = slot_valid(idx[k], a.rows);
        const uint16_t *row = a.gemm2 + (ok ? static_cast<int64_t>(idx[k]) * a.ld : 0);
#pragma unroll
        for (int c = 0; c < CPT; ++c)
            q[k][c] = ok ? ld_nc_na_16(row + (tid + c * NT) * kChunkElems) : make_uint4(0, 0, 0, 0);
    }

    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);

    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (!slot_valid(idx[k], a.rows)) continue;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            float x[8];
            unpack8(q[k][c], x);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w[k], x[j], acc[c][j]);
        }
    }

    const bool before = a.before != 0;
    float ss = warp_sum(prenorm<CPT>(acc, g, before));
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) tot += red[i];
    const float r = rsqrtf(__fmaf_rn(tot, 1.0f / kTpHidden, a.eps));

    scale_store<CPT, NT>(acc, g, before, r, a.out + t * kTpHidden, tid);
}

// ---------------------------------------------------------------------------
// decode sizes: a cluster of C CTAs per token

template <int C, int WK>
__global__ void __launch_bounds__(kChunksPerRow / C) tp_cluster_kernel(const TpArgs a) {
    constexpr int NT = kChunksPerRow / C;  // one chunk per thread
    constexpr int NW = NT / 32;
    __shared__ float red[NW];
    __shared__ float part;

    const uint32_t rank = cluster_ctarank();
    const int64_t t = blockIdx.x / C;
    const int tid = threadIdx.x;
    const int chunk = static_cast<int>(rank) * NT + tid;

    pdl_wait();
    pdl_trigger();  // the next call's CTAs may be scheduled now (they still wait for this grid)
    int idx[8];
    float w[8];
    load_route<WK>(a, t, idx, w);

    uint4 q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool ok = slot_valid(idx[k], a.rows);
        const uint16_t *row = a.gemm2 + (ok ? static_cast<int64_t>(idx[k]) * a.ld : 0);
        q[k] = ok ? ld_nc_na_16(row + chunk * kChunkElems) : make_uint4(0, 0, 0, 0);
    }
    float g[1][8];
    load_gain(a, chunk, g[0]);

    float acc[1][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[0][j] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (!slot_valid(idx[k], a.rows)) continue;
        float x[8];
        unpack8(q[k], x);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[0][j] = __fmaf_rn(w[k], x[j], acc[0][j]);
    }

    const bool before = a.before != 0;
    const float ss = warp_sum(prenorm<1>(acc, g, before));
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < NW; ++i) p += red[i];
        part = p;
    }
    cluster_barrier();  // every CTA's partial is written and visible
    float tot = 0.f;
    const uint32_t part_addr = smem_u32(&part);
#pragma unroll
    for (int r = 0; r < C; ++r) tot += ld_dsmem_f32(part_addr, r);  // same order in every CTA
    const float r = rsqrtf(__fmaf_rn(tot, 1.0f / kTpHidden, a.eps));

    scale_store<1, 1>(acc, g, before, r, a.out + t * kTpHidden, chunk);
    // no CTA leaves while another may still read its `part`; every value read
    // from a peer has been used above, and no peer reads the stores, so the
    // arrive is relaxed (4-6 % less per decode call than release / acquire)
    cluster_barrier_exit();
}

// ---------------------------------------------------------------------------
// one CTA per token, rows staged in shared memory by bulk copies

// Thread 0 copies every valid row of the token (8 KB each) into its slot of a
// 64 KB shared-memory buffer with one-dimensional bulk copies, each completing
// on the row's own mbarrier; the data in flight holds no registers, so three CTAs
// (192 KB of rows) can be in flight per SM.  Every thread then waits on the
// barrier, reads its CPT chunks of each valid row from shared memory and runs
// the same FMA chain and epilogue as the register kernel.
constexpr int kBulkCPT = 2;                      // 256 threads
constexpr int kBulkThreads = kChunksPerRow / kBulkCPT;
constexpr int kBulkSmem = kTpTopK * kTpRowBytes;  // 64 KB of rows

template <int WK>
__global__ void __launch_bounds__(kBulkThreads)
    tp_token_bulk_kernel(const TpArgs a) {
    constexpr int NT = kBulkThreads, NW = NT / 32, CPT = kBulkCPT;
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[8];
    __shared__ float red[NW];

    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    const uint32_t rows_base = smem_u32(rows_smem);

    pdl_wait();
    int idx[8];
    float w[8];
    load_route<WK>(a, t, idx, w);
    uint32_t mask = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) mask |= (slot_valid(idx[k], a.rows) ? 1u : 0u) << k;

    // one mbarrier per row: the reduction starts on a row as soon as it lands
    if (tid == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mbar_init(smem_u32(&bars[k]), 1);
        fence_mbar_init();
        const uint64_t policy = policy_evict_first();
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if ((mask >> k) & 1u) {
                const uint32_t b = smem_u32(&bars[k]);
                mbar_arrive_expect_tx(b, kTpRowBytes);
                bulk_copy_g2s_hint(rows_base + k * kTpRowBytes,
                                   a.gemm2 + static_cast<int64_t>(idx[k]) * a.ld, kTpRowBytes, b,
                                   policy);
            }
    }
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);
    __syncthreads();  // the barriers are initialised before anyone waits on them

    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (!((mask >> k) & 1u)) continue;
        const uint32_t b = smem_u32(&bars[k]);
        if (!mbar_wait(b, 0u, a.timeout_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            ok = false;
            (void)mbar_wait(b, 0u, a.timeout_ns);  // bounded: the copy may land, or not, before exit
        }
        uint4 q[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) q[c] = lds_16(rows_base + k * kTpRowBytes + (tid + c * NT) * kChunkBytes);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            float x[8];
            unpack8(q[c], x);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(w[k], x[j], acc[c][j]);
        }
    }

    const bool before = a.before != 0;
    const float ss = warp_sum(prenorm<CPT>(acc, g, before));
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) tot += red[i];
    const float r = rsqrtf(__fmaf_rn(tot, 1.0f / kTpHidden, a.eps));
    if (ok) scale_store<CPT, NT>(acc, g, before, r, a.out + t * kTpHidden, tid);
}

// The same staged kernel for launches of five waves and more, with several
// tokens in each of the first `groups` CTAs.  CTA b < groups takes
// kBulkTokensPerCta consecutive tokens, the CTAs after it one token each (the
// last waves of the launch).  A CTA with more tokens loads the next token's
// route while the current token's rows land, and once every thread has read
// those rows it puts the next token's rows in flight into the same buffer
// before the current token's norm and stores, so the route's DRAM round trip
// and the epilogue of all but its last token overlap row traffic.  One-token
// CTAs at the end keep the drain of a launch as short as with one token per
// CTA.  Each token's arithmetic is that of tp_token_bulk_kernel: the same bits.
constexpr int kBulkTokensPerCta = 3;
constexpr int kBulkSingleWaves = 2;  // waves of one-token CTAs at the end

template <int WK>
__global__ void __launch_bounds__(kBulkThreads, 3)
    tp_token_bulk_multi_kernel(const TpArgs a, const int64_t groups) {
    constexpr int NT = kBulkThreads, NW = NT / 32, CPT = kBulkCPT;
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[8];
    __shared__ float red[2][NW];

    const int64_t b = blockIdx.x;
    const bool grouped = b < groups;
    int64_t t = grouped ? kBulkTokensPerCta * b : (kBulkTokensPerCta - 1) * groups + b;
    const int ntok = grouped ? kBulkTokensPerCta : 1;
    const int tid = threadIdx.x;
    const uint32_t rows_base = smem_u32(rows_smem);

    pdl_wait();
    int idx[8];
    float w[8];
    load_route<WK>(a, t, idx, w);
    uint32_t mask = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) mask |= (slot_valid(idx[k], a.rows) ? 1u : 0u) << k;

    // one mbarrier per row: the reduction starts on a row as soon as it lands
    // (thread 0 initialises the barriers and arms them, in its own order)
    auto issue = [&](const int (&ix)[8], uint32_t m) {
        const uint64_t policy = policy_evict_first();
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if ((m >> k) & 1u) {
                const uint32_t bb = smem_u32(&bars[k]);
                mbar_arrive_expect_tx(bb, kTpRowBytes);
                bulk_copy_g2s_hint(rows_base + k * kTpRowBytes,
                                   a.gemm2 + static_cast<int64_t>(ix[k]) * a.ld, kTpRowBytes, bb,
                                   policy);
            }
    };
    if (tid == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mbar_init(smem_u32(&bars[k]), 1);
        fence_mbar_init();
        issue(idx, mask);
    }
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);
    __syncthreads();  // the barriers are initialised before anyone waits on them

    const bool before = a.before != 0;
    uint32_t parity = 0;  // bit k: the phase of bars[k] the next wait is for
    for (int j = 0; j < ntok; ++j, ++t) {
        int nidx[8];
        float nw[8];
        uint32_t nmask = 0;
        if (j + 1 < ntok) {  // the next token's route, while this token's rows land
            load_route<WK>(a, t + 1, nidx, nw);
#pragma unroll
            for (int k = 0; k < 8; ++k) nmask |= (slot_valid(nidx[k], a.rows) ? 1u : 0u) << k;
        }
        float acc[CPT][8];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
        bool ok = true;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (!((mask >> k) & 1u)) continue;
            const uint32_t bb = smem_u32(&bars[k]);
            const uint32_t ph = (parity >> k) & 1u;
            if (!mbar_wait(bb, ph, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                ok = false;
                (void)mbar_wait(bb, ph, a.timeout_ns);  // bounded: the copy may land, or not, before exit
            }
            uint4 q[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) q[c] = lds_16(rows_base + k * kTpRowBytes + (tid + c * NT) * kChunkBytes);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float x[8];
                unpack8(q[c], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[c][e] = __fmaf_rn(w[k], x[e], acc[c][e]);
            }
        }
        parity ^= mask;  // the barriers armed for this token moved to their next phase
        bool more = false;
        if (j + 1 < ntok) {
            // every thread has read the buffer, and none gave up waiting: the
            // next token's rows go in flight before this token's epilogue
            more = !__syncthreads_or(!ok);
            if (more && tid == 0) {
                fence_proxy_async_smem();  // the reads above come before the copies
                issue(nidx, nmask);
            }
        }
        float *rd = red[j & 1];  // alternate: a slow warp may still read the last one
        const float ss = warp_sum(prenorm<CPT>(acc, g, before));
        if ((tid & 31) == 0) rd[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < NW; ++i) tot += rd[i];
        const float r = rsqrtf(__fmaf_rn(tot, 1.0f / kTpHidden, a.eps));
        if (ok) scale_store<CPT, NT>(acc, g, before, r, a.out + t * kTpHidden, tid);
        if (!more) break;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            idx[k] = nidx[k];
            w[k] = nw[k];
        }
        mask = nmask;
    }
}

// ---------------------------------------------------------------------------
// data movement alone (a measurement aid; not part of the operation)

// The memory traffic of the hidden-4096 finalize without its arithmetic: one
// CTA per token loads the route (index and weight of each slot), copies each
// valid row into shared memory (one bulk copy and one mbarrier per row, as
// tp_token_bulk_kernel), every thread reads its chunks of each row back, and
// the token's output row goes out with the same streaming stores.  What it
// stores is the XOR of the words read (the weights included), so the compiler
// keeps every load and no floating-point work is done.  Timed on the same
// buffers as the finalize, it shows what the reduction, the norm and the
// scheduling of the finalize kernels cost on top of the bytes they move.
template <int WK>
__global__ void __launch_bounds__(kBulkThreads, 3) tp_data_movement_kernel(const TpArgs a) {
    constexpr int NT = kBulkThreads, CPT = kBulkCPT;
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[8];

    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    const uint32_t rows_base = smem_u32(rows_smem);

    pdl_wait();
    int idx[8];
    float w[8];
    load_route<WK>(a, t, idx, w);
    uint32_t mask = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) mask |= (slot_valid(idx[k], a.rows) ? 1u : 0u) << k;
    if (tid == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mbar_init(smem_u32(&bars[k]), 1);
        fence_mbar_init();
        const uint64_t policy = policy_evict_first();
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if ((mask >> k) & 1u) {
                const uint32_t b = smem_u32(&bars[k]);
                mbar_arrive_expect_tx(b, kTpRowBytes);
                bulk_copy_g2s_hint(rows_base + k * kTpRowBytes,
                                   a.gemm2 + static_cast<int64_t>(idx[k]) * a.ld, kTpRowBytes, b,
                                   policy);
            }
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them

    uint4 x[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) x[c] = make_uint4(0u, 0u, 0u, 0u);
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (!((mask >> k) & 1u)) continue;
        const uint32_t b = smem_u32(&bars[k]);
        if (!mbar_wait(b, 0u, a.timeout_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            ok = false;
            (void)mbar_wait(b, 0u, a.timeout_ns);  // bounded: the copy may land, or not, before exit
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const uint4 q = lds_16(rows_base + k * kTpRowBytes + (tid + c * NT) * kChunkBytes);
            x[c].x ^= q.x ^ __float_as_uint(w[k]);
            x[c].y ^= q.y;
            x[c].z ^= q.z;
            x[c].w ^= q.w;
        }
    }
    if (ok) {
#pragma unroll
        for (int c = 0; c < CPT; ++c)
            st_cs_16(a.out + t * kTpHidden + static_cast<int64_t>(tid + c * NT) * kChunkElems, x[c]);
    }
}

// ---------------------------------------------------------------------------
// any hidden / top-k: one CTA per token, valid rows staged in pieces

// Warp 0 reads the route (lane k holds slot k) and compacts the valid slots in
// ascending k into shared memory; up to `rows_per_piece` valid rows at a time
// go into the staging buffer with one bulk copy per row.  The first piece
// leaves as soon as the route is known, before the CTA's barrier and the
// norm_weight loads, each of its rows issued by the lane of
// its slot; thread 0 issues the later pieces.  Each thread
// owns CPT 16-byte chunks of the H columns.  Same arithmetic as the
// specialised kernels: FP32 FMA over valid slots in ascending k, then the
// RMSNorm epilogue with the mean over the H columns.
template <int WK>
__device__ __forceinline__ float load_weight(const void *weights, int64_t i) {
    if constexpr (WK == kWeightBF16) {
        const uint32_t b = __ldg(static_cast<const unsigned short *>(weights) + i);
        return __uint_as_float(b << 16);
    } else if constexpr (WK == kWeightPacked) {
        return bf16_lo(static_cast<uint32_t>(__ldg(static_cast<const int32_t *>(weights) + i)));
    } else {
        return __ldg(static_cast<const float *>(weights) + i);
    }
}

// Launch bounds: up to 512 threads with two CTAs per SM for CPT 2; up to
// 1024 threads (hidden 256 x odd) for CPT 1.
template <int CPT>
constexpr int generic_max_threads() { return CPT == 2 ? 512 : 1024; }
template <int CPT>
constexpr int generic_min_blocks() { return CPT == 2 ? 2 : 1; }

// PER_ROW: one mbarrier per buffered row, so the reduction starts on a row as
// soon as it lands; otherwise one per piece (small rows with many slots, where
// a wait per row costs more than it overlaps).
template <int CPT, int WK, bool PER_ROW>
__global__ void __launch_bounds__(generic_max_threads<CPT>(), generic_min_blocks<CPT>())
    tp_generic_bulk_kernel(const TpArgs a, const int rows_per_piece) {
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[PER_ROW ? 32 : 1];
    __shared__ float red[32];
    __shared__ float w_s[32];
    __shared__ int idx_s[32];
    __shared__ int order_s[32];
    __shared__ int nvalid_s;

    const int NT = blockDim.x;
    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x;
    const int H = a.hidden, K = a.top_k;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2;
    const uint32_t base = smem_u32(rows_smem);
    const uint32_t bar_addr = smem_u32(&bars[0]);

    // Copy valid rows p0..p0+n-1 (in ascending slot order) into the buffer
    // (thread 0, for the pieces after the first).
    auto issue_piece = [&](int p0, int n) {
        const uint64_t policy = policy_evict_first();
        if (!PER_ROW) mbar_arrive_expect_tx(bar_addr, n * row_bytes);
        for (int r = 0; r < n; ++r) {
            const uint32_t b = PER_ROW ? smem_u32(&bars[r]) : bar_addr;
            if (PER_ROW) mbar_arrive_expect_tx(b, row_bytes);
            bulk_copy_g2s_hint(base + r * row_bytes,
                               a.gemm2 + static_cast<int64_t>(idx_s[order_s[p0 + r]]) * a.ld,
                               row_bytes, b, policy);
        }
    };

    pdl_wait();
    if (tid < 32) {
        int i = -1;
        if (tid < K) i = __ldg(a.idx + t * K + tid);
        const bool valid = tid < K && slot_valid(i, a.rows);
        // the weight (of a valid slot only) is requested before the rows, so
        // that it does not queue behind them, and used after the copies are issued
        const float w = valid ? load_weight<WK>(a.weights, t * K + tid) : 0.f;
        const unsigned mask = __ballot_sync(0xffffffffu, valid);
        const int nv = __popc(mask);
        const int rank = __popc(mask & ((1u << tid) - 1u));
        idx_s[tid] = i;
        if (valid) order_s[rank] = tid;
        if (PER_ROW) {
            // the lane of the rank-th valid slot owns row `rank` of the first
            // piece: it initialises and arms that row's mbarrier and copies its
            // own row, so the first piece's copies leave together
            if (valid && rank < rows_per_piece) {
                const uint32_t b = smem_u32(&bars[rank]);
                mbar_init(b, 1);
                fence_mbar_init();
                mbar_arrive_expect_tx(b, row_bytes);
                bulk_copy_g2s_hint(base + rank * row_bytes, a.gemm2 + static_cast<int64_t>(i) * a.ld,
                                   row_bytes, b, policy_evict_first());
            }
            if (tid == 0) nvalid_s = nv;
        } else {  // small rows, many slots: one mbarrier for the piece, each
                  // row still issued by the lane of its slot
            if (tid == 0) {
                mbar_init(bar_addr, 1);
                fence_mbar_init();
                nvalid_s = nv;
                if (nv > 0) mbar_arrive_expect_tx(bar_addr, (nv < rows_per_piece ? nv : rows_per_piece) * row_bytes);
            }
            __syncwarp();
            if (valid && rank < rows_per_piece)
                bulk_copy_g2s_hint(base + rank * row_bytes, a.gemm2 + static_cast<int64_t>(i) * a.ld,
                                   row_bytes, bar_addr, policy_evict_first());
        }
        w_s[tid] = w;
    }
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);
    __syncthreads();

    const int nvalid = nvalid_s;
    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

    bool ok = true;
    uint32_t phase = 0;
    for (int p0 = 0; p0 < nvalid; p0 += rows_per_piece, phase ^= 1u) {
        const int n = nvalid - p0 < rows_per_piece ? nvalid - p0 : rows_per_piece;
        if (tid == 0 && p0 > 0) {
            fence_proxy_async_smem();  // earlier reads of the buffer come first
            issue_piece(p0, n);
        }
        for (int r = 0; r < n; ++r) {
            if (PER_ROW || r == 0) {
                const uint32_t b = PER_ROW ? smem_u32(&bars[r]) : bar_addr;
                if (!mbar_wait(b, phase, a.timeout_ns)) {
                    atomicOr(a.status, kStatusWaitTimeout);
                    ok = false;
                    (void)mbar_wait(b, phase, a.timeout_ns);  // bounded: the copies may land, or not, before exit
                }
            }
            const float w = w_s[order_s[p0 + r]];
            const uint32_t row = base + r * row_bytes;
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
        if (p0 + rows_per_piece < nvalid) __syncthreads();  // the next piece reuses the buffer
    }

    const bool before = a.before != 0;
    const float ss = warp_sum(prenorm<CPT>(acc, g, before));
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    const int nw = NT >> 5;
    for (int i = 0; i < nw; ++i) tot += red[i];
    const float r = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(H)), a.eps));
    if (!ok) return;
    uint16_t *out_row = a.out + t * H;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float s = __fmul_rn(acc[c][j], r);
            y[j] = before ? s : __fmul_rn(s, g[c][j]);
        }
        st_cs_16(out_row + static_cast<int64_t>(tid + c * NT) * kChunkElems, pack8_rn(y));
    }
}

// The generic staged kernel with several tokens per CTA, for launches of five
// waves and more whose tokens fit the buffer in one piece (top_k <= the rows
// per piece) with a barrier per row.  As in tp_token_bulk_multi_kernel, CTA
// b < groups takes n consecutive tokens and the CTAs of the last two waves u
// each; the buffer holds SLOTS tokens' rows (one or two), each in the rank
// order of its valid slots.  Warp 0 loads the route of the token SLOTS ahead
// while the current rows land, and once every thread has read them the lane
// of each of its valid slots copies its row into the freed buffer slot, before
// the current token's norm and stores.  The compacted weights of a token are
// stored by the lanes that copy its rows, before they arm the row barriers,
// whose release orders them before every reader's acquire.  Each token's
// arithmetic is that of tp_generic_bulk_kernel: the same bits.
constexpr int kGenericTokensPerCta = 3;  // n = 3 x SLOTS
constexpr int kGenericSingleWaves = 2;   // waves of u-token CTAs at the end

struct GenericLayout {
    int64_t groups;  // CTAs b < groups take n tokens, the later ones u (the last one fewer)
    int n;
    int u;
    int slots;       // tokens whose rows the buffer holds at once (0: not this kernel)
};

template <int CPT, int WK, int SLOTS>
__global__ void __launch_bounds__(generic_max_threads<CPT>(), generic_min_blocks<CPT>())
    tp_generic_bulk_multi_kernel(const TpArgs a, const GenericLayout lay) {
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[32];  // buffer slot s, rank r at s * top_k + r
    __shared__ float red[2][32];
    __shared__ float wc_s[32];     // weights of the valid slots, same index
    __shared__ int nvalid_s[SLOTS];

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
        const int64_t left = a.num_tokens - t0;
        cnt = left < lay.u ? static_cast<int>(left) : lay.u;
    }
    const int H = a.hidden, K = a.top_k;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2;
    const uint32_t slot_bytes = row_bytes * static_cast<uint32_t>(K);
    const uint32_t base = smem_u32(rows_smem);

    // warp 0, lane k: slot k of a token's route -- record its weight by rank and
    // copy its row into buffer slot `bs` at its rank (all of a token's valid rows fit)
    auto place = [&](int i, bool valid, float w, int bs) {
        const unsigned mask = __ballot_sync(0xffffffffu, valid);
        const int rank = __popc(mask & ((1u << tid) - 1u));
        if (valid) {
            wc_s[bs * K + rank] = w;
            const uint32_t bb = smem_u32(&bars[bs * K + rank]);
            mbar_arrive_expect_tx(bb, row_bytes);
            bulk_copy_g2s_hint(base + bs * slot_bytes + rank * row_bytes,
                               a.gemm2 + static_cast<int64_t>(i) * a.ld, row_bytes, bb,
                               policy_evict_first());
        }
        if (tid == 0) nvalid_s[bs] = __popc(mask);
    };
    if (tid < SLOTS * K) {
        mbar_init(smem_u32(&bars[tid]), 1);
        fence_mbar_init();
    }
    pdl_wait();
    if (tid < 32) {
        __syncwarp();
        const int first = cnt < SLOTS ? cnt : SLOTS;
        for (int bs = 0; bs < first; ++bs) {
            int i = -1;
            if (tid < K) i = __ldg(a.idx + (t0 + bs) * K + tid);
            const bool valid = tid < K && slot_valid(i, a.rows);
            // the weight (of a valid slot only) is requested before the copy
            const float w = valid ? load_weight<WK>(a.weights, (t0 + bs) * K + tid) : 0.f;
            place(i, valid, w, bs);
        }
    }
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);
    __syncthreads();

    const bool before = a.before != 0;
    uint32_t parity = 0;  // bit s * top_k + r: the phase of that barrier the next wait is for
    int bs = 0;
    for (int j = 0; j < cnt; ++j) {
        const int64_t t = t0 + j;
        const int nvalid = nvalid_s[bs];
        const bool refill = j + SLOTS < cnt;
        int ni = -1;  // warp 0: the route of the token SLOTS ahead, while this token's rows land
        bool nvalid_slot = false;
        float nwt = 0.f;
        if (refill && tid < 32) {
            if (tid < K) ni = __ldg(a.idx + (t + SLOTS) * K + tid);
            nvalid_slot = tid < K && slot_valid(ni, a.rows);
            nwt = nvalid_slot ? load_weight<WK>(a.weights, (t + SLOTS) * K + tid) : 0.f;
        }
        float acc[CPT][8];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
        bool ok = true;
        for (int r = 0; r < nvalid; ++r) {
            const int q = bs * K + r;
            const uint32_t bb = smem_u32(&bars[q]);
            const uint32_t ph = (parity >> q) & 1u;
            if (!mbar_wait(bb, ph, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                ok = false;
                (void)mbar_wait(bb, ph, a.timeout_ns);  // bounded: the copy may land, or not, before exit
            }
            const float w = wc_s[q];
            const uint32_t row = base + bs * slot_bytes + r * row_bytes;
            uint4 qd[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) qd[c] = lds_16(row + (tid + c * NT) * kChunkBytes);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float x[8];
                unpack8(qd[c], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[c][e] = __fmaf_rn(w, x[e], acc[c][e]);
            }
        }
        // the barriers of ranks 0..nvalid-1 of this buffer slot moved on
        parity ^= (nvalid >= 32 ? 0xffffffffu : ((1u << nvalid) - 1u)) << (bs * K);
        bool more = true;
        if (refill) {
            // every thread has read this buffer slot and none gave up waiting:
            // the token SLOTS ahead goes in flight into it before this epilogue
            more = !__syncthreads_or(!ok);
            if (more && tid < 32) {
                fence_proxy_async_smem();  // the reads above come before the copies
                place(ni, nvalid_slot, nwt, bs);
            }
        }
        const int rb = j & 1;  // alternate: a slow warp may still read the last one
        const float ss = warp_sum(prenorm<CPT>(acc, g, before));
        if ((tid & 31) == 0) red[rb][tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        const int nw = NT >> 5;
        for (int i = 0; i < nw; ++i) tot += red[rb][i];
        const float r = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(H)), a.eps));
        if (ok) {
            uint16_t *out_row = a.out + t * H;
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float sv = __fmul_rn(acc[c][e], r);
                    y[e] = before ? sv : __fmul_rn(sv, g[c][e]);
                }
                st_cs_16(out_row + static_cast<int64_t>(tid + c * NT) * kChunkElems, pack8_rn(y));
            }
        }
        if (!more) break;
        if (SLOTS > 1 && ++bs == SLOTS) bs = 0;
    }
}

// ---------------------------------------------------------------------------
// small hidden (256..1024): one warp per token, four tokens per CTA

// Each warp owns one token and up to 16 KB of shared memory: lane k reads slot
// k of the route, the valid slots are compacted with a ballot, and up to
// `rows_per_piece` valid rows at a time are copied with one bulk copy per row,
// each issued by the lane of its slot (one mbarrier per warp and piece).  The
// RMS is a warp reduction, so warps never wait for one another.  Each lane
// owns CPW 16-byte chunks (hidden = 256 CPW).
// Two tokens per CTA (measured against four and eight: the same or faster at
// every hidden size, 5 % at 256 x 32 and 4 % at 768; eight up to 25 % slower).
template <int CPW>
constexpr int warp_tokens_per_cta() { return 2; }
constexpr int kWarpSliceBytes = 16384;  // 8 rows of the largest warp-path row (2 KB)

template <int CPW, int WK>
__global__ void __launch_bounds__(32 * warp_tokens_per_cta<CPW>())
    tp_warp_bulk_kernel(const TpArgs a, const int rows_per_piece) {
    constexpr int kWarpTokensPerCta = warp_tokens_per_cta<CPW>();
    // each warp's slice holds rows_per_piece rows (at most kWarpSliceBytes)
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[kWarpTokensPerCta];
    constexpr int H = 256 * CPW;
    constexpr uint32_t row_bytes = H * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpTokensPerCta + warp;
    if (t >= a.num_tokens) return;
    const int K = a.top_k;
    const uint32_t base = smem_u32(rows_smem) + warp * rows_per_piece * row_bytes;
    const uint32_t bar = smem_u32(&bars[warp]);

    pdl_wait();
    int my_idx = -1;
    if (lane < K) my_idx = __ldg(a.idx + t * K + lane);
    const bool valid = lane < K && slot_valid(my_idx, a.rows);
    const float my_w = valid ? load_weight<WK>(a.weights, t * K + lane) : 0.f;
    const unsigned mask = __ballot_sync(0xffffffffu, valid);
    const int nvalid = __popc(mask);
    const int my_rank = __popc(mask & ((1u << lane) - 1u));
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    float g[CPW][8];
#pragma unroll
    for (int c = 0; c < CPW; ++c) load_gain(a, lane + c * 32, g[c]);
    __syncwarp();

    float acc[CPW][8];
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;
    bool ok = true;
    uint32_t phase = 0;
    unsigned rest = mask;  // valid slots not yet consumed, ascending
    for (int p0 = 0; p0 < nvalid; p0 += rows_per_piece, phase ^= 1u) {
        const int n = nvalid - p0 < rows_per_piece ? nvalid - p0 : rows_per_piece;
        if (p0 > 0) fence_proxy_async_smem();  // earlier reads of the slice come first
        if (lane == 0) mbar_arrive_expect_tx(bar, n * row_bytes);
        __syncwarp();
        // the lane of each valid slot in the piece copies its own row (all at once)
        if (valid && my_rank >= p0 && my_rank < p0 + n)
            bulk_copy_g2s_hint(base + (my_rank - p0) * row_bytes,
                               a.gemm2 + static_cast<int64_t>(my_idx) * a.ld, row_bytes, bar,
                               policy_evict_first());
        if (!mbar_wait(bar, phase, a.timeout_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            ok = false;
            (void)mbar_wait(bar, phase, a.timeout_ns);  // bounded: the copies may land, or not, before exit
        }
        for (int r = 0; r < n; ++r) {
            const int k = __ffs(rest) - 1;
            rest &= rest - 1;
            const float w = __shfl_sync(0xffffffffu, my_w, k);
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

    const bool before = a.before != 0;
    const float tot = warp_sum(prenorm<CPW>(acc, g, before));
    const float r = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(H)), a.eps));
    if (!ok) return;
    scale_store<CPW, 32>(acc, g, before, r, a.out + t * H, lane);
}

// The warp-per-token kernel with several tokens per warp, for launches of five
// waves of resident warps and more whose tokens fit the warp's slice in one
// piece (top_k <= rows per piece).  Warp u < groups (counted over the grid,
// two per CTA) takes kWarpMultiTokens consecutive tokens, the warps of the
// last two waves one each.  A warp loads the next token's route while the
// current rows land and, once its lanes have read them, copies the next
// token's rows into its slice before the current token's norm and stores.  The
// warp's mbarrier moves to its next phase only for tokens with valid rows.
// Each token's arithmetic is that of tp_warp_bulk_kernel: the same bits.
constexpr int kWarpMultiTokens = 3;
constexpr int kWarpSingleWaves = 2;  // waves of one-token warps at the end

template <int CPW, int WK>
__global__ void __launch_bounds__(32 * warp_tokens_per_cta<CPW>())
    tp_warp_bulk_multi_kernel(const TpArgs a, const int rows_per_piece, const int64_t groups) {
    constexpr int kWarpTokensPerCta = warp_tokens_per_cta<CPW>();
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bars[kWarpTokensPerCta];
    constexpr int H = 256 * CPW;
    constexpr uint32_t row_bytes = H * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * kWarpTokensPerCta + warp;
    const bool grouped = u < groups;
    int64_t t = grouped ? kWarpMultiTokens * u : (kWarpMultiTokens - 1) * groups + u;
    if (t >= a.num_tokens) return;
    const int ntok = grouped ? kWarpMultiTokens : 1;
    const int K = a.top_k;
    const uint32_t base = smem_u32(rows_smem) + warp * rows_per_piece * row_bytes;
    const uint32_t bar = smem_u32(&bars[warp]);

    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // this warp's copies of token `tok`'s valid rows, each by the lane of its
    // slot, into the slice position of its rank
    auto issue = [&](int i, bool valid, unsigned mask) {
        const int nv = __popc(mask);
        if (nv == 0) return;
        if (lane == 0) mbar_arrive_expect_tx(bar, nv * row_bytes);
        __syncwarp();
        if (valid)
            bulk_copy_g2s_hint(base + __popc(mask & ((1u << lane) - 1u)) * row_bytes,
                               a.gemm2 + static_cast<int64_t>(i) * a.ld, row_bytes, bar,
                               policy_evict_first());
    };

    pdl_wait();
    int my_idx = -1;
    if (lane < K) my_idx = __ldg(a.idx + t * K + lane);
    bool valid = lane < K && slot_valid(my_idx, a.rows);
    float my_w = valid ? load_weight<WK>(a.weights, t * K + lane) : 0.f;
    unsigned mask = __ballot_sync(0xffffffffu, valid);
    issue(my_idx, valid, mask);
    float g[CPW][8];
#pragma unroll
    for (int c = 0; c < CPW; ++c) load_gain(a, lane + c * 32, g[c]);

    const bool before = a.before != 0;
    uint32_t phase = 0;
    for (int j = 0; j < ntok; ++j, ++t) {
        int nidx = -1;  // the next token's route, while this token's rows land
        bool nvalid = false;
        float nw = 0.f;
        if (j + 1 < ntok) {
            if (lane < K) nidx = __ldg(a.idx + (t + 1) * K + lane);
            nvalid = lane < K && slot_valid(nidx, a.rows);
            nw = nvalid ? load_weight<WK>(a.weights, (t + 1) * K + lane) : 0.f;
        }
        float acc[CPW][8];
#pragma unroll
        for (int c = 0; c < CPW; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
        bool ok = true;
        if (mask != 0u) {
            if (!mbar_wait(bar, phase, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                ok = false;
                (void)mbar_wait(bar, phase, a.timeout_ns);  // bounded: the copies may land, or not, before exit
            }
            phase ^= 1u;
            unsigned rest = mask;
            const int n = __popc(mask);
            for (int r = 0; r < n; ++r) {
                const int k = __ffs(rest) - 1;
                rest &= rest - 1;
                const float w = __shfl_sync(0xffffffffu, my_w, k);
                const uint32_t row = base + r * row_bytes;
                uint4 q[CPW];
#pragma unroll
                for (int c = 0; c < CPW; ++c) q[c] = lds_16(row + (lane + c * 32) * kChunkBytes);
#pragma unroll
                for (int c = 0; c < CPW; ++c) {
                    float x[8];
                    unpack8(q[c], x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[c][e] = __fmaf_rn(w, x[e], acc[c][e]);
                }
            }
        }
        bool more = false;
        if (j + 1 < ntok) {
            // every lane has read the slice, and none gave up waiting: the next
            // token's rows go in flight before this token's epilogue
            more = __all_sync(0xffffffffu, ok);
            if (more) {
                fence_proxy_async_smem();  // the reads above come before the copies
                const unsigned nmask = __ballot_sync(0xffffffffu, nvalid);
                issue(nidx, nvalid, nmask);
                my_idx = nidx;
                valid = nvalid;
                mask = nmask;
            }
        }
        const float tot = warp_sum(prenorm<CPW>(acc, g, before));
        const float r = rsqrtf(__fadd_rn(__fdiv_rn(tot, static_cast<float>(H)), a.eps));
        if (ok) scale_store<CPW, 32>(acc, g, before, r, a.out + t * H, lane);
        if (!more) break;
        my_w = nw;
    }
}

// 2 chunks per thread when that leaves at least 128 threads (hidden 2048 and
// up, an even number of 256-column groups), else 1.  At hidden 2048-3584 two
// chunks per thread measured 1-7 % faster than one (fewer threads wait on each
// row's barrier).
int generic_cpt(int hidden) { return ((hidden / 256) % 2 == 0 && hidden / 16 >= 128) ? 2 : 1; }

// Shared memory for one CTA's rows, sized so that two CTAs fit an SM (1 KB
// system reservation and up to 1 KB of static shared memory per CTA included).
int generic_budget(int smem_per_sm) { return smem_per_sm / 2 - 1024 - 1024; }

// Rows per piece: at least 8 (a whole token at top_k <= 8), otherwise pieces
// sized so that eight CTAs fit an SM, and never more than half an SM's shared
// memory.  With many slots, small pieces keep more tokens in flight per SM and
// let one piece's reduction overlap other CTAs' copies: 2048 x 32 1.04 of the
// copy peak against 0.80 with pieces of half an SM, 1536 x 32 1.00 against
// 0.73, 2560 x 24 1.03 against 0.85; the 8-slot sizes do not change.
int generic_rows(int smem_per_sm, int top_k, int hidden) {
    int rows = (smem_per_sm / 8 - 2048) / (hidden * 2);
    if (rows < 8) rows = 8;
    const int half = generic_budget(smem_per_sm) / (hidden * 2);
    if (rows > half) rows = half;
    return rows < 1 ? 1 : (rows > top_k ? top_k : rows);
}

template <typename Kern>
cudaError_t set_dyn_smem(Kern k, int bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t prepare_tp_kernels(int smem_optin, int smem_per_sm) {
    const int budget = generic_budget(smem_per_sm);
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_kernel<kWeightBF16>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_kernel<kWeightFP32>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_kernel<kWeightPacked>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_multi_kernel<kWeightBF16>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_multi_kernel<kWeightFP32>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_token_bulk_multi_kernel<kWeightPacked>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_data_movement_kernel<kWeightBF16>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_data_movement_kernel<kWeightFP32>, kBulkSmem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_data_movement_kernel<kWeightPacked>, kBulkSmem);
    constexpr int warp_smem1 = kWarpSliceBytes * warp_tokens_per_cta<1>();
    constexpr int warp_smem = kWarpSliceBytes * warp_tokens_per_cta<2>();  // CPW 2..4
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<1, kWeightBF16>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<1, kWeightFP32>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<1, kWeightPacked>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<2, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<2, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<2, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<3, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<3, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<3, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<4, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<4, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_kernel<4, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<1, kWeightBF16>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<1, kWeightFP32>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<1, kWeightPacked>, warp_smem1);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<2, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<2, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<2, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<3, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<3, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<3, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<4, kWeightBF16>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<4, kWeightFP32>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_warp_bulk_multi_kernel<4, kWeightPacked>, warp_smem);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightBF16, false>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightFP32, false>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightPacked, false>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightBF16, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightFP32, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<1, kWeightPacked, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<2, kWeightBF16, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<2, kWeightFP32, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_kernel<2, kWeightPacked, true>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<1, kWeightBF16, 1>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<1, kWeightFP32, 1>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<1, kWeightPacked, 1>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightBF16, 1>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightFP32, 1>, budget);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightPacked, 1>, budget);
    // two token slots: up to the CTA's whole share at the one-token kernel's occupancy
    const int two = smem_optin < smem_per_sm - 2048 ? smem_optin : smem_per_sm - 2048;
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightBF16, 2>, two);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightFP32, 2>, two);
    if (e == cudaSuccess) e = set_dyn_smem(tp_generic_bulk_multi_kernel<2, kWeightPacked, 2>, two);
    return e;
}

cudaError_t tp_blocks_per_sm(int *bulk, int *token_cta) {
    int multi = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        bulk, tp_token_bulk_kernel<kWeightFP32>, kBulkThreads, kBulkSmem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &multi, tp_token_bulk_multi_kernel<kWeightFP32>, kBulkThreads, kBulkSmem);
    if (e == cudaSuccess && multi < *bulk) *bulk = multi;  // both kernels' waves: the smaller
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(token_cta, tp_token_cta_kernel<1, kWeightFP32>,
                                                          kChunksPerRow, 0);
    return e;
}

cudaError_t launch_tp_token_cta(const TpArgs &a, int wk, cudaStream_t s) {
    constexpr int CPT = 1;
    const dim3 grid(static_cast<unsigned>(a.num_tokens)), block(kChunksPerRow / CPT);
    const bool p = a.programmatic;
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_token_cta_kernel<CPT, kWeightBF16>, grid, block, 0, s, 1, p, a);
        case kWeightPacked: return launch_ex(tp_token_cta_kernel<CPT, kWeightPacked>, grid, block, 0, s, 1, p, a);
        default: return launch_ex(tp_token_cta_kernel<CPT, kWeightFP32>, grid, block, 0, s, 1, p, a);
    }
}

cudaError_t launch_tp_cluster(const TpArgs &a, int wk, cudaStream_t s) {
    constexpr int C = 8;
    const dim3 grid(static_cast<unsigned>(a.num_tokens * C)), block(kChunksPerRow / C);
    const bool p = a.programmatic;
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_cluster_kernel<C, kWeightBF16>, grid, block, 0, s, C, p, a);
        case kWeightPacked: return launch_ex(tp_cluster_kernel<C, kWeightPacked>, grid, block, 0, s, C, p, a);
        default: return launch_ex(tp_cluster_kernel<C, kWeightFP32>, grid, block, 0, s, C, p, a);
    }
}

int64_t tp_bulk_groups(int64_t num_tokens, int64_t resident) {
    const int64_t n = kBulkTokensPerCta, singles = int64_t{kBulkSingleWaves} * resident;
    if (resident <= 0 || num_tokens < singles + n * resident) return 0;
    int64_t groups = (num_tokens - singles) / n;
    // a partial wave of multi-token CTAs that would end after the one-token CTAs
    // have run out (it starts one wave of multi-token CTAs late) is dropped
    const int64_t r = groups % resident;
    if (r != 0 && n * (resident - r) > singles) groups -= r;
    return groups;
}

cudaError_t launch_tp_bulk(const TpArgs &a, int wk, int resident_ctas, cudaStream_t s) {
    const int64_t groups = tp_bulk_groups(a.num_tokens, resident_ctas);
    const bool p = a.programmatic;
    const dim3 block(kBulkThreads);
    if (groups == 0) {
        const dim3 grid(static_cast<unsigned>(a.num_tokens));
        switch (wk) {
            case kWeightBF16: return launch_ex(tp_token_bulk_kernel<kWeightBF16>, grid, block, kBulkSmem, s, 1, p, a);
            case kWeightPacked: return launch_ex(tp_token_bulk_kernel<kWeightPacked>, grid, block, kBulkSmem, s, 1, p, a);
            default: return launch_ex(tp_token_bulk_kernel<kWeightFP32>, grid, block, kBulkSmem, s, 1, p, a);
        }
    }
    const dim3 grid(static_cast<unsigned>(a.num_tokens - (kBulkTokensPerCta - 1) * groups));
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_token_bulk_multi_kernel<kWeightBF16>, grid, block, kBulkSmem, s, 1, p, a, groups);
        case kWeightPacked: return launch_ex(tp_token_bulk_multi_kernel<kWeightPacked>, grid, block, kBulkSmem, s, 1, p, a, groups);
        default: return launch_ex(tp_token_bulk_multi_kernel<kWeightFP32>, grid, block, kBulkSmem, s, 1, p, a, groups);
    }
}

cudaError_t launch_tp_data_movement(const TpArgs &a, int wk, cudaStream_t s) {
    const bool p = a.programmatic;
    const dim3 grid(static_cast<unsigned>(a.num_tokens)), block(kBulkThreads);
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_data_movement_kernel<kWeightBF16>, grid, block, kBulkSmem, s, 1, p, a);
        case kWeightPacked: return launch_ex(tp_data_movement_kernel<kWeightPacked>, grid, block, kBulkSmem, s, 1, p, a);
        default: return launch_ex(tp_data_movement_kernel<kWeightFP32>, grid, block, kBulkSmem, s, 1, p, a);
    }
}

template <int CPT, bool PER_ROW>
static cudaError_t launch_generic_cpt(const TpArgs &a, int wk, int rows, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.num_tokens)), block(a.hidden / 8 / CPT);
    const size_t bytes = static_cast<size_t>(rows) * a.hidden * 2;
    const bool p = a.programmatic;
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_generic_bulk_kernel<CPT, kWeightBF16, PER_ROW>, grid, block, bytes, s, 1, p, a, rows);
        case kWeightPacked: return launch_ex(tp_generic_bulk_kernel<CPT, kWeightPacked, PER_ROW>, grid, block, bytes, s, 1, p, a, rows);
        default: return launch_ex(tp_generic_bulk_kernel<CPT, kWeightFP32, PER_ROW>, grid, block, bytes, s, 1, p, a, rows);
    }
}

// One mbarrier per row for rows of 4 KB and more (hidden >= 2048), and for
// smaller rows when top_k <= 16 (hidden 1280-1792 x 8: 0.99 of the copy peak
// against 0.94-0.96 with one barrier per piece); with more slots of small rows
// one barrier per piece measured faster (1536 x 32: 167.6 against 173.3 us).
constexpr int kPerRowMinHidden = 2048;
constexpr int kPerRowMaxTopK = 16;

// Rows per piece of the warp-per-token kernels: at least 8 and up to 8 KB of
// them (hidden 256 x 32: 16 rows, 0.95 of the copy peak against 0.82 with 32;
// hidden 1024: 8 rows, 16 KB)
static int warp_rows(int hidden, int top_k) {
    int rows = 8192 / (hidden * 2);
    if (rows < 8) rows = 8;
    return rows > top_k ? top_k : rows;
}

template <int CPW>
static int warp_multi_per_sm(int wk, size_t bytes) {
    constexpr int threads = 32 * warp_tokens_per_cta<CPW>();
    int n = 0;
    cudaError_t e;
    switch (wk) {
        case kWeightBF16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_warp_bulk_multi_kernel<CPW, kWeightBF16>, threads, bytes); break;
        case kWeightPacked: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_warp_bulk_multi_kernel<CPW, kWeightPacked>, threads, bytes); break;
        default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_warp_bulk_multi_kernel<CPW, kWeightFP32>, threads, bytes); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Multi-token warps of a warp-per-token launch (0: one token per warp).
template <int CPW>
static int64_t warp_groups(int64_t num_tokens, int top_k, int wk, int num_sms) {
    constexpr int H = 256 * CPW;
    const int rows = warp_rows(H, top_k);
    if (top_k > rows || num_sms <= 0) return 0;  // a token's rows in one piece
    const size_t bytes = static_cast<size_t>(rows) * H * 2 * warp_tokens_per_cta<CPW>();
    const int64_t resident =
        int64_t{warp_multi_per_sm<CPW>(wk, bytes)} * warp_tokens_per_cta<CPW>() * num_sms;
    const int64_t n = kWarpMultiTokens, singles = int64_t{kWarpSingleWaves} * resident;
    if (resident <= 0 || num_tokens < singles + n * resident) return 0;
    int64_t groups = (num_tokens - singles) / n;
    const int64_t r = groups % resident;  // drop a partial wave that would outlast the rest
    if (r != 0 && n * (resident - r) > singles) groups -= r;
    return groups;
}

template <int CPW>
static cudaError_t launch_warp_cpw(const TpArgs &a, int wk, int num_sms, cudaStream_t s) {
    constexpr int kWarpTokensPerCta = warp_tokens_per_cta<CPW>();
    const int rows = warp_rows(a.hidden, a.top_k);
    const dim3 block(32 * kWarpTokensPerCta);
    const size_t bytes = static_cast<size_t>(rows) * a.hidden * 2 * kWarpTokensPerCta;
    const bool p = a.programmatic;
    const int64_t groups = warp_groups<CPW>(a.num_tokens, a.top_k, wk, num_sms);
    if (groups > 0) {
        const int64_t units = a.num_tokens - (kWarpMultiTokens - 1) * groups;
        const dim3 mgrid(static_cast<unsigned>((units + kWarpTokensPerCta - 1) / kWarpTokensPerCta));
        switch (wk) {
            case kWeightBF16: return launch_ex(tp_warp_bulk_multi_kernel<CPW, kWeightBF16>, mgrid, block, bytes, s, 1, p, a, rows, groups);
            case kWeightPacked: return launch_ex(tp_warp_bulk_multi_kernel<CPW, kWeightPacked>, mgrid, block, bytes, s, 1, p, a, rows, groups);
            default: return launch_ex(tp_warp_bulk_multi_kernel<CPW, kWeightFP32>, mgrid, block, bytes, s, 1, p, a, rows, groups);
        }
    }
    const dim3 grid(static_cast<unsigned>((a.num_tokens + kWarpTokensPerCta - 1) / kWarpTokensPerCta));
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_warp_bulk_kernel<CPW, kWeightBF16>, grid, block, bytes, s, 1, p, a, rows);
        case kWeightPacked: return launch_ex(tp_warp_bulk_kernel<CPW, kWeightPacked>, grid, block, bytes, s, 1, p, a, rows);
        default: return launch_ex(tp_warp_bulk_kernel<CPW, kWeightFP32>, grid, block, bytes, s, 1, p, a, rows);
    }
}

template <int CPT, int SLOTS>
static int generic_multi_per_sm(int wk, int threads, size_t bytes) {
    int n = 0;
    cudaError_t e;
    switch (wk) {
        case kWeightBF16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_multi_kernel<CPT, kWeightBF16, SLOTS>, threads, bytes); break;
        case kWeightPacked: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_multi_kernel<CPT, kWeightPacked, SLOTS>, threads, bytes); break;
        default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_multi_kernel<CPT, kWeightFP32, SLOTS>, threads, bytes); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// CTAs per SM of the one-token generic kernel (with a barrier per row).
template <int CPT>
static int generic_one_per_sm(int wk, int threads, size_t bytes) {
    int n = 0;
    cudaError_t e;
    switch (wk) {
        case kWeightBF16: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_kernel<CPT, kWeightBF16, true>, threads, bytes); break;
        case kWeightPacked: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_kernel<CPT, kWeightPacked, true>, threads, bytes); break;
        default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tp_generic_bulk_kernel<CPT, kWeightFP32, true>, threads, bytes); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

int64_t tp_warp_groups(int64_t num_tokens, int hidden, int top_k, int wk, int num_sms) {
    switch (hidden) {
        case 256: return warp_groups<1>(num_tokens, top_k, wk, num_sms);
        case 512: return warp_groups<2>(num_tokens, top_k, wk, num_sms);
        case 768: return warp_groups<3>(num_tokens, top_k, wk, num_sms);
        case 1024: return warp_groups<4>(num_tokens, top_k, wk, num_sms);
        default: return 0;
    }
}

// Tokens per CTA: n for the first `groups` CTAs, u for the later ones, from
// five waves of resident CTAs; a partial wave of n-token CTAs that would end
// after the u-token CTAs have run out (it starts one wave late) is dropped.
static GenericLayout generic_groups(int64_t num_tokens, int slots, int64_t resident) {
    GenericLayout lay = {0, 0, 0, 0};
    if (resident <= 0) return lay;
    int64_t u = num_tokens / (4 * resident);  // later CTAs small enough for about four waves
    if (u > slots) u = slots;
    if (u < 1) u = 1;
    const int64_t n = int64_t{kGenericTokensPerCta} * slots, singles = kGenericSingleWaves * u * resident;
    if (num_tokens < singles + n * resident) return lay;
    int64_t groups = (num_tokens - singles) / n;
    const int64_t r = groups % resident;
    if (r != 0 && n * (resident - r) > singles) groups -= r;
    lay.groups = groups;
    lay.n = static_cast<int>(n);
    lay.u = static_cast<int>(u);
    lay.slots = slots;
    return lay;
}

// The several-tokens layout of a generic launch (slots 0: one token per CTA).
// Two token slots where the tokens are small (at hidden 4096..7168 and top_k
// 1..3: 4-14 % faster than one slot; 2048 x 2 +3.5 %): only when two whole
// tokens fit the shared memory a CTA gets at the one-token kernel's
// occupancy, the two-slot kernel keeps that occupancy, and the launch is long
// enough for n-token CTAs (two-token CTAs alone measured 5 % slower than one
// slot at 3000 x 7168 x 4).  Otherwise one slot, three tokens per CTA.
static GenericLayout generic_layout(int64_t num_tokens, int hidden, int top_k, int wk,
                                    int smem_per_sm, int num_sms) {
    GenericLayout none = {0, 0, 0, 0};
    if (hidden <= 1024 || num_sms <= 0) return none;  // the warp-per-token kernel
    const int rows = generic_rows(smem_per_sm, top_k, hidden);
    if (top_k > rows) return none;  // a token's rows in one piece (with a barrier per row)
    if (num_tokens < int64_t{kGenericTokensPerCta + kGenericSingleWaves} * num_sms) return none;
    const int cpt = generic_cpt(hidden);
    const int threads = hidden / 8 / cpt;
    const int64_t token_bytes = int64_t{top_k} * hidden * 2;
    if (cpt == 2 && 2 * top_k <= 32) {
        const int occ_one = generic_one_per_sm<2>(wk, threads, static_cast<size_t>(token_bytes));
        const int occ_two = generic_multi_per_sm<2, 2>(wk, threads, 0);
        if (occ_one > 0 && occ_two >= occ_one && smem_per_sm / occ_one - 2048 >= 2 * token_bytes) {
            const int per_sm = generic_multi_per_sm<2, 2>(wk, threads, static_cast<size_t>(2 * token_bytes));
            const GenericLayout two = generic_groups(num_tokens, 2, int64_t{per_sm} * num_sms);
            if (two.groups > 0) return two;
        }
    }
    const size_t bytes = static_cast<size_t>(rows) * hidden * 2;
    const int per_sm = cpt == 2 ? generic_multi_per_sm<2, 1>(wk, threads, bytes)
                                : generic_multi_per_sm<1, 1>(wk, threads, bytes);
    const GenericLayout one = generic_groups(num_tokens, 1, int64_t{per_sm} * num_sms);
    return one.groups > 0 ? one : none;
}

int64_t tp_generic_groups(int64_t num_tokens, int hidden, int top_k, int wk, int smem_per_sm,
                          int num_sms) {
    return generic_layout(num_tokens, hidden, top_k, wk, smem_per_sm, num_sms).groups;
}

template <int CPT>
static cudaError_t launch_generic_multi(const TpArgs &a, int wk, const GenericLayout &lay,
                                       cudaStream_t s) {
    const int64_t ctas = lay.groups + (a.num_tokens - int64_t{lay.n} * lay.groups + lay.u - 1) / lay.u;
    const dim3 grid(static_cast<unsigned>(ctas));
    const dim3 block(a.hidden / 8 / CPT);
    const size_t bytes = static_cast<size_t>(lay.slots) * a.top_k * a.hidden * 2;
    const bool p = a.programmatic;
    if constexpr (CPT == 2) {  // two slots only with two chunks per thread
        if (lay.slots == 2) {
            switch (wk) {
                case kWeightBF16: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightBF16, 2>, grid, block, bytes, s, 1, p, a, lay);
                case kWeightPacked: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightPacked, 2>, grid, block, bytes, s, 1, p, a, lay);
                default: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightFP32, 2>, grid, block, bytes, s, 1, p, a, lay);
            }
        }
    }
    switch (wk) {
        case kWeightBF16: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightBF16, 1>, grid, block, bytes, s, 1, p, a, lay);
        case kWeightPacked: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightPacked, 1>, grid, block, bytes, s, 1, p, a, lay);
        default: return launch_ex(tp_generic_bulk_multi_kernel<CPT, kWeightFP32, 1>, grid, block, bytes, s, 1, p, a, lay);
    }
}

cudaError_t launch_tp_generic(const TpArgs &a, int wk, int smem_per_sm, int num_sms,
                              cudaStream_t s) {
    // hidden 256..1024: one warp per token
    switch (a.hidden) {
        case 256: return launch_warp_cpw<1>(a, wk, num_sms, s);
        case 512: return launch_warp_cpw<2>(a, wk, num_sms, s);
        case 768: return launch_warp_cpw<3>(a, wk, num_sms, s);
        case 1024: return launch_warp_cpw<4>(a, wk, num_sms, s);
        default: break;
    }
    const int rows = generic_rows(smem_per_sm, a.top_k, a.hidden);
    const GenericLayout lay = generic_layout(a.num_tokens, a.hidden, a.top_k, wk, smem_per_sm, num_sms);
    if (lay.slots > 0) {
        if (generic_cpt(a.hidden) == 2) return launch_generic_multi<2>(a, wk, lay, s);
        return launch_generic_multi<1>(a, wk, lay, s);
    }
    if (generic_cpt(a.hidden) == 2) return launch_generic_cpt<2, true>(a, wk, rows, s);  // hidden >= 2048
    if (a.hidden >= kPerRowMinHidden || a.top_k <= kPerRowMaxTopK)
        return launch_generic_cpt<1, true>(a, wk, rows, s);
    return launch_generic_cpt<1, false>(a, wk, rows, s);
}

}  // namespace mf
