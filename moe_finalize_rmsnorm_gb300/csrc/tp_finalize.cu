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
//   tp_token_bulk_kernel one CTA per token; thread 0 stages the token's valid
//                        rows in shared memory with 1-D bulk copies
//                        (cp.async.bulk) completing on one mbarrier, so no
//                        registers are held by data in flight and three
//                        CTAs (192 KB of rows) fit per SM.
//
// Every wait on an mbarrier is bounded (TpArgs::timeout_ns); a wait that gives
// up ORs kStatusWaitTimeout into the device status word and the kernel returns.

#include "common.cuh"
#include "kernels.h"

namespace mf {
namespace {

constexpr int kChunksPerRow = kTpHidden / kChunkElems;  // 512

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
// one CTA per token, rows staged in shared memory by bulk copies

// Thread 0 copies every valid row of the token (8 KB each) into its slot of a
// 64 KB shared-memory buffer with one-dimensional bulk copies that complete on
// a single mbarrier; the data in flight holds no registers, so three CTAs
// (192 KB of rows) can be in flight per SM.  Every thread then waits on the
// barrier, reads its CPT chunks of each valid row from shared memory and runs
// the same FMA chain and epilogue as the register kernel.
constexpr int kBulkCPT = 2;                      // 256 threads
constexpr int kBulkThreads = kChunksPerRow / kBulkCPT;
constexpr int kBulkSmem = kTpTopK * kTpRowBytes;  // 64 KB of rows

template <bool BF16W>
__global__ void __launch_bounds__(kBulkThreads)
    tp_token_bulk_kernel(const TpArgs a) {
    constexpr int NT = kBulkThreads, NW = NT / 32, CPT = kBulkCPT;
    extern __shared__ __align__(128) uint8_t rows_smem[];
    __shared__ uint64_t bar;
    __shared__ float red[NW];

    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    const uint32_t rows_base = smem_u32(rows_smem);
    const uint32_t bar_addr = smem_u32(&bar);

    int idx[8];
    float w[8];
    load_route<BF16W>(a, t, idx, w);
    uint32_t mask = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) mask |= (slot_valid(idx[k], a.rows) ? 1u : 0u) << k;

    if (tid == 0) {
        mbar_init(bar_addr, 1);
        fence_mbar_init();
        const uint64_t policy = policy_evict_first();
        mbar_arrive_expect_tx(bar_addr, static_cast<uint32_t>(__popc(mask)) * kTpRowBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if ((mask >> k) & 1u)
                bulk_copy_g2s_hint(rows_base + k * kTpRowBytes,
                                   a.gemm2 + static_cast<int64_t>(idx[k]) * a.ld, kTpRowBytes,
                                   bar_addr, policy);
    }
    float g[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) load_gain(a, tid + c * NT, g[c]);
    __syncthreads();  // the barrier is initialised before anyone waits on it

    bool ok = mbar_wait(bar_addr, 0u, a.timeout_ns);
    if (!ok) {
        atomicOr(a.status, kStatusWaitTimeout);
        ok = mbar_wait(bar_addr, 0u, a.timeout_ns);  // let copies in flight land before exit
    }

    float acc[CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (!((mask >> k) & 1u)) continue;
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

}  // namespace

cudaError_t prepare_tp_kernels(int smem_optin) {
    (void)smem_optin;
    cudaError_t e = cudaFuncSetAttribute(tp_token_bulk_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tp_token_bulk_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
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

cudaError_t launch_tp_bulk(const TpArgs &a, bool bf16_weights, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.num_tokens)), block(kBulkThreads);
    if (bf16_weights)
        tp_token_bulk_kernel<true><<<grid, block, kBulkSmem, s>>>(a);
    else
        tp_token_bulk_kernel<false><<<grid, block, kBulkSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mf
