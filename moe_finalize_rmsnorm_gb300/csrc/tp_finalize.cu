// Finalize + RMSNorm kernels for hidden 4096, top-k 8 (sm_103a).
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
//   tp_ring_kernel       persistent, one CTA per SM: a producer thread streams
//                        the valid rows of the CTA's tokens into a ring of
//                        8 KB shared-memory slots with 1-D bulk copies
//                        (cp.async.bulk, completion on per-slot mbarriers);
//                        consumer warps read each slot once, FMA into FP32
//                        registers, release the slot, and finish each token
//                        with the RMSNorm epilogue and 16-byte streaming stores.
//                        Up to ~28 rows (224 KB) are in flight per SM.
//
// Every wait on an mbarrier is bounded (TpArgs::timeout_ns); a wait that gives
// up ORs kStatusWaitTimeout into the device status word and the kernel returns.

#include "common.cuh"
#include "kernels.h"

namespace mf {
namespace {

constexpr int kChunksPerRow = kTpHidden / kChunkElems;  // 512
constexpr uint32_t kMetaLast = 1u;   // slot holds the token's last valid row
constexpr uint32_t kMetaEmpty = 2u;  // token has no valid row; slot carries no data

// Load the 8 route entries of token t (same address across the block: the
// loads are broadcasts).
template <bool BF16W>
__device__ __forceinline__ void load_route(const TpArgs &a, int64_t t, int (&idx)[8],
                                           float (&w)[8]) {
    const int4 *ip = reinterpret_cast<const int4 *>(a.idx + t * kTpTopK);
    const int4 i0 = __ldg(ip), i1 = __ldg(ip + 1);
    idx[0] = i0.x; idx[1] = i0.y; idx[2] = i0.z; idx[3] = i0.w;
    idx[4] = i1.x; idx[5] = i1.y; idx[6] = i1.z; idx[7] = i1.w;
    if constexpr (BF16W) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(
            static_cast<const uint16_t *>(a.weights) + t * kTpTopK));
        unpack8(q, w);
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

template <int CPT, bool BF16W>
__global__ void __launch_bounds__(kChunksPerRow / CPT)
    tp_token_cta_kernel(const TpArgs a) {
    constexpr int NT = kChunksPerRow / CPT;
    constexpr int NW = NT / 32;
    __shared__ float red[NW];

    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;

    int idx[8];
    float w[8];
    load_route<BF16W>(a, t, idx, w);

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

template <int C, bool BF16W>
__global__ void __launch_bounds__(kChunksPerRow / C) tp_cluster_kernel(const TpArgs a) {
    constexpr int NT = kChunksPerRow / C;  // one chunk per thread
    constexpr int NW = NT / 32;
    __shared__ float red[NW];
    __shared__ float part;

    const uint32_t rank = cluster_ctarank();
    const int64_t t = blockIdx.x / C;
    const int tid = threadIdx.x;
    const int chunk = static_cast<int>(rank) * NT + tid;

    int idx[8];
    float w[8];
    load_route<BF16W>(a, t, idx, w);

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
    cluster_barrier();  // no CTA leaves while another may still read its `part`
}

// ---------------------------------------------------------------------------
// persistent bulk-copy ring

struct RingMeta {
    float w;
    uint32_t flags;
};

struct RingLayout {
    int slots;
    size_t bytes;
    // offsets from the dynamic shared memory base
    size_t full, empty, redbar, meta, red;
};

__host__ __device__ inline RingLayout ring_layout(int slots, int slot_bytes, int consumer_warps) {
    RingLayout L;
    L.slots = slots;
    size_t off = static_cast<size_t>(slots) * slot_bytes;
    L.full = off;   off += sizeof(uint64_t) * slots;
    L.empty = off;  off += sizeof(uint64_t) * slots;
    L.redbar = off; off += sizeof(uint64_t) * 2;
    L.meta = off;   off += sizeof(RingMeta) * slots;
    L.red = off;    off += sizeof(float) * 2 * consumer_warps;
    L.bytes = off;
    return L;
}

template <int CPT, bool BF16W>
__global__ void __launch_bounds__(kChunksPerRow / CPT + 32, 1)
    tp_ring_kernel(const TpArgs a, const int slots) {
    constexpr int NC = kChunksPerRow / CPT;  // consumer threads
    constexpr int NCW = NC / 32;
    extern __shared__ __align__(1024) uint8_t smem[];
    const RingLayout L = ring_layout(slots, kTpRowBytes, NCW);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *redbar = reinterpret_cast<uint64_t *>(smem + L.redbar);
    RingMeta *meta = reinterpret_cast<RingMeta *>(smem + L.meta);
    float *red = reinterpret_cast<float *>(smem + L.red);
    const uint32_t ring_base = smem_u32(smem);

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

    const int64_t T = a.num_tokens;
    const int64_t stride = gridDim.x;

    if (tid >= NC) {
        // ------------------------------------------------------ producer
        if (tid != NC) return;
        const uint64_t policy = policy_evict_first();
        uint32_t pos = 0;
        int64_t t = blockIdx.x;
        if (t >= T) return;
        int nidx[8];
        float nw[8];
        load_route<BF16W>(a, t, nidx, nw);
        bool ok = true;
        for (; t < T && ok; t += stride) {
            int idx[8];
            float w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) { idx[k] = nidx[k]; w[k] = nw[k]; }
            if (t + stride < T) load_route<BF16W>(a, t + stride, nidx, nw);  // prefetch
            uint32_t mask = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) mask |= (slot_valid(idx[k], a.rows) ? 1u : 0u) << k;
            if (mask == 0) {
                const int s = pos % slots;
                const uint32_t ph = (pos / slots) & 1u;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.timeout_ns)) { ok = false; break; }
                meta[s] = RingMeta{0.f, kMetaLast | kMetaEmpty};
                mbar_arrive(smem_u32(&full[s]));
                ++pos;
                continue;
            }
            const int last = 31 - __clz(mask);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (!((mask >> k) & 1u)) continue;
                const int s = pos % slots;
                const uint32_t ph = (pos / slots) & 1u;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.timeout_ns)) { ok = false; break; }
                meta[s] = RingMeta{w[k], k == last ? kMetaLast : 0u};
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, kTpRowBytes);
                bulk_copy_g2s_hint(ring_base + static_cast<uint32_t>(s) * kTpRowBytes,
                                   a.gemm2 + static_cast<int64_t>(idx[k]) * a.ld, kTpRowBytes, fb,
                                   policy);
                ++pos;
            }
        }
        if (!ok) {
            atomicOr(a.status, kStatusWaitTimeout);
            // drain: wait (bounded) for the copies this thread issued
            const uint32_t first = pos > static_cast<uint32_t>(slots) ? pos - slots : 0u;
            for (uint32_t p = first; p < pos; ++p)
                (void)mbar_wait(smem_u32(&full[p % slots]), (p / slots) & 1u, a.timeout_ns);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31, warp = tid >> 5;
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NC, g[c]);
    const bool before = a.before != 0;

    uint32_t pos = 0, titer = 0;
    for (int64_t t = blockIdx.x; t < T; t += stride, ++titer) {
        float acc[CPT][8];
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;

        for (;;) {
            const int s = pos % slots;
            const uint32_t ph = (pos / slots) & 1u;
            if (!mbar_wait(smem_u32(&full[s]), ph, a.timeout_ns)) {
                atomicOr(a.status, kStatusWaitTimeout);
                return;
            }
            const RingMeta m = meta[s];
            if (!(m.flags & kMetaEmpty)) {
                const uint32_t slot = ring_base + static_cast<uint32_t>(s) * kTpRowBytes;
                uint4 q[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) q[c] = lds_16(slot + (tid + c * NC) * kChunkBytes);
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float x[8];
                    unpack8(q[c], x);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[c][j] = __fmaf_rn(m.w, x[j], acc[c][j]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            ++pos;
            if (m.flags & kMetaLast) break;
        }

        const float ss = warp_sum(prenorm<CPT>(acc, g, before));
        const int b = titer & 1;
        if (lane == 0) {
            red[b * NCW + warp] = ss;
            mbar_arrive(smem_u32(&redbar[b]));
        }
        if (!mbar_wait(smem_u32(&redbar[b]), (titer >> 1) & 1u, a.timeout_ns)) {
            atomicOr(a.status, kStatusWaitTimeout);
            return;
        }
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < NCW; ++i) tot += red[b * NCW + i];
        const float r = rsqrtf(__fmaf_rn(tot, 1.0f / kTpHidden, a.eps));
        scale_store<CPT, NC>(acc, g, before, r, a.out + t * kTpHidden, tid);
    }
}

constexpr int kRingCPT = 2;  // 256 consumer threads + 1 producer warp

int ring_slots(int smem_optin) {
    const int ncw = kChunksPerRow / kRingCPT / 32;
    int slots = 1;
    while (ring_layout(slots + 1, kTpRowBytes, ncw).bytes <= static_cast<size_t>(smem_optin))
        ++slots;
    return slots;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

}  // namespace

cudaError_t prepare_tp_kernels(int smem_optin) {
    const int slots = ring_slots(smem_optin);
    const size_t bytes = ring_layout(slots, kTpRowBytes, kChunksPerRow / kRingCPT / 32).bytes;
    cudaError_t e = set_smem(tp_ring_kernel<kRingCPT, false>, bytes);
    if (e == cudaSuccess) e = set_smem(tp_ring_kernel<kRingCPT, true>, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tp_cluster_kernel<16, false>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tp_cluster_kernel<16, true>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

cudaError_t launch_tp_token_cta(const TpArgs &a, bool bf16_weights, cudaStream_t s) {
    constexpr int CPT = 1;
    const dim3 grid(static_cast<unsigned>(a.num_tokens)), block(kChunksPerRow / CPT);
    if (bf16_weights)
        tp_token_cta_kernel<CPT, true><<<grid, block, 0, s>>>(a);
    else
        tp_token_cta_kernel<CPT, false><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

template <int C>
static cudaError_t launch_cluster_c(const TpArgs &a, bool bf16_weights, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.num_tokens * C));
    cfg.blockDim = dim3(kChunksPerRow / C);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bf16_weights) return cudaLaunchKernelEx(&cfg, tp_cluster_kernel<C, true>, a);
    return cudaLaunchKernelEx(&cfg, tp_cluster_kernel<C, false>, a);
}

cudaError_t launch_tp_cluster(const TpArgs &a, bool bf16_weights, cudaStream_t s) {
    return launch_cluster_c<8>(a, bf16_weights, s);
}

cudaError_t launch_tp_ring(const TpArgs &a, bool bf16_weights, int num_sms, int smem_optin,
                           cudaStream_t s) {
    const int slots = ring_slots(smem_optin);
    const size_t bytes = ring_layout(slots, kTpRowBytes, kChunksPerRow / kRingCPT / 32).bytes;
    const int64_t grid = a.num_tokens < num_sms ? a.num_tokens : num_sms;
    const dim3 block(kChunksPerRow / kRingCPT + 32);
    if (bf16_weights)
        tp_ring_kernel<kRingCPT, true><<<static_cast<unsigned>(grid), block, bytes, s>>>(a, slots);
    else
        tp_ring_kernel<kRingCPT, false><<<static_cast<unsigned>(grid), block, bytes, s>>>(a, slots);
    return cudaGetLastError();
}

}  // namespace mf
