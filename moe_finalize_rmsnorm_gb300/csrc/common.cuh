// Device helpers shared by the finalize kernels (sm_103a).
//
// BF16 <-> FP32 conversions, 16-byte global loads/stores, mbarrier and
// bulk-copy (cp.async.bulk) wrappers with bounded waits, and cluster/DSMEM
// primitives.  All inline PTX here is hand-written.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mf {

// Bits OR-ed into the library's device status word.
constexpr unsigned kStatusWaitTimeout = 1u;

// 16 bytes = 8 BF16 values.
constexpr int kChunkElems = 8;
constexpr int kChunkBytes = 16;

// ---------------------------------------------------------------------------
// BF16 <-> FP32 (a BF16 value is the upper half of a binary32)

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &q, float (&f)[8]) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x);
    f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z);
    f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
}

__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ uint4 pack8_rn(const float (&f)[8]) {
    return make_uint4(pack2_rn(f[0], f[1]), pack2_rn(f[2], f[3]), pack2_rn(f[4], f[5]),
                      pack2_rn(f[6], f[7]));
}

// Round each value to BF16 and return the rounded value as FP32 (exact).
__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------------------
// global memory

// Read-only 16-byte load that does not allocate in L1 (each gathered row
// element is used once).
__device__ __forceinline__ uint4 ld_nc_na_16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Coherent 16-byte load that does not allocate in L1: for data this kernel
// may itself overwrite (the residual op may write hidden into its residual
// buffer), where the read-only (.nc) path is not allowed.
__device__ __forceinline__ uint4 ld_na_16(const void *p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Streaming 16-byte store (written once, not re-read by this kernel).
__device__ __forceinline__ void st_cs_16(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// shared memory, mbarriers and bulk copies

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the other threads and to the
// asynchronous (bulk-copy) proxy; follow with a CTA barrier.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier to complete, for at most
// `limit_ns` nanoseconds of wall time.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u && globaltimer_ns() - start > limit_ns) return false;
    }
}

// Order this thread's earlier generic-proxy shared-memory accesses (and, after
// a CTA barrier, the other threads') before later bulk-copy writes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on mbarrier `bar`, with an L2 eviction-priority
// policy (evict-first for rows read once).  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                                   uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 lds_16(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr)
                 : "memory");
    return r;
}

// ---------------------------------------------------------------------------
// clusters and distributed shared memory

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

// The same barrier with a relaxed arrive: it orders none of this thread's
// earlier memory operations for the other CTAs, so it does not wait for
// outstanding global stores to drain.  For the end of a cluster kernel, where
// the barrier only keeps a CTA's shared memory alive until every peer has
// consumed what it read from it (the values read must already be in use).
__device__ __forceinline__ void cluster_barrier_exit() {
    asm volatile(
        "barrier.cluster.arrive.relaxed.aligned;\n\t"
        "barrier.cluster.wait.aligned;" ::
            : "memory");
}

// Load a float from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch

// Wait until the grids this one depends on have completed and their memory is
// visible.  Every kernel calls it before its first global-memory access; it
// returns at once when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next grid in the stream be scheduled (its pdl_wait still holds it
// until this grid has completed).  Only the decode-size cluster kernel calls
// it, right after its own dependency wait (1.75 against 1.92 us per one-token
// call in a CUDA graph; 2.05 us without the trigger).  A grid also triggers
// when it completes; on kernels with many small CTAs the explicit trigger costs
// more than it gains (15 us on 65536 one-warp CTAs), and in the register
// kernel at 16-128 tokens it measured within 2 % either way.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launch with an optional cluster width and, when `programmatic`, the
// programmatic stream serialisation attribute (the kernel may be scheduled
// while its predecessor in the stream finishes; its pdl_wait orders memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, unsigned cluster_x, bool programmatic,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (programmatic) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace mf
