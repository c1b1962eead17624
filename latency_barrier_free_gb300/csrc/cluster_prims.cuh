// cluster_prims.cuh -- device helpers of the kernels that run one virtual
// rank per CTA of a thread-block cluster (cluster.cu, coll.cu): cluster
// identity, distributed shared memory addressing, split cluster barriers,
// st.async pushes and bulk copies that complete the receiver's mbarrier,
// bounded mbarrier waits.  Every wait here is bounded by a Waiter (prims.cuh).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "prims.cuh"

namespace rra {
namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}

__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];"
                 :
                 : "r"(raddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
                 : "memory");
}

// Bulk copy (the TMA engine, no tensor map) of `bytes` (a multiple of 16;
// both addresses 16-byte aligned) from global memory into the shared memory
// of every CTA of the cluster set in `mask`, at the same offset `dst` in
// each; each destination's mbarrier at offset `bar` counts the bytes.
__device__ __forceinline__ void bulk_g2s_multicast(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                                   uint16_t mask) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1], %2, [%3], "
        "%4;"
        :
        : "r"(dst), "l"(src), "r"(bytes), "r"(bar), "h"(mask)
        : "memory");
}

// Bulk copy (the TMA engine) of `bytes` (a multiple of 16; both addresses
// 16-byte aligned) from this CTA's shared memory `src` to global memory
// `dst`, in the issuing thread's bulk group.  Data that an earlier bulk copy
// or st.async wrote into `src` is read once the mbarrier that counted it has
// completed and fence_proxy_async_smem() has run.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :
                 : "l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

// The issuing thread's bulk copies to global memory, committed and waited
// for until their writes are done (so shared memory may be released and the
// outputs are complete when the CTA exits).
__device__ __forceinline__ void bulk_s2g_commit_wait() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this CTA's earlier shared-memory accesses before later accesses by
// the async proxy (bulk copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;" : "=l"(state) : "r"(bar), "r"(bytes) : "memory");
}

// Arrive (release, cluster scope) on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" : : "r"(cluster_bar) : "memory");
}

// Bounded wait of all threads on one phase of a local mbarrier.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, Waiter& w) {
    while (!mbar_try_wait(bar, parity))
        if (waiter_expired(w)) return false;
    return true;
}

}  // namespace
}  // namespace rra
