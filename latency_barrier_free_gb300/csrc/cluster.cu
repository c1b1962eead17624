// cluster.cu -- one-shot push AllReduce through distributed shared memory.
//
// "Every Microsecond Matters", Sec. III-A (one-shot, push) and Sec. IV (data
// arrival as the only synchronisation), restated for what one GB300 offers
// below L2: the CTAs of a thread-block cluster sit on one GPC and can store
// into each other's shared memory.  A cluster holds one CTA per virtual rank
// for one slice of the message; CTA r's shared memory is rank r's window for
// that slice.  Each CTA pushes its input slice into slot [r] of every peer
// with st.async, which also completes the receiver's mbarrier transaction
// count; the receiver waits on its own mbarrier -- the arrival of the bytes
// is the signal -- and adds the N slots in rank order (bit-identical to the
// other one-shot kernels).
//
// Shared memory and mbarriers live only as long as a launch, so no epoch or
// flag state persists between calls and nothing needs resetting.  The price
// is two hardware cluster barriers per call (barrier.cluster, within one GPC):
// after the mbarrier initialisation, so that no CTA stores into a peer's
// barrier before it exists, and before exit, so that no CTA leaves while a
// peer may still store into its shared memory.  Neither orders data; the
// data readiness is the mbarrier's transaction count alone.  Clusters do not
// wait on each other, so any number of them may run in waves.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "prims.cuh"
#include "rra_internal.h"

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

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];"
                 :
                 : "r"(raddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(256) oneshot_cluster_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [nranks][per_cta] payload vectors
    __shared__ __align__(8) uint64_t bar;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint64_t t_start = globaltimer_ns();
    const int N = p.nranks;
    const int r = (int)cluster_ctarank();
    const uint32_t slice = cluster_id();
    const uint32_t P = p.per_cta;
    const uint32_t pos0 = slice * P;
    const uint32_t npos = min(P, p.nvec - pos0);
    // first input vector and the injected-fault word, both in flight at once
    uint4 first = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < npos) first = load_input<T>(p.send[r], pos0 + threadIdx.x, p.count);
    const int32_t drop = (int32_t)ld_relaxed_u32(&p.ctrl->drop_rank);

    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(my_bar), "r"(1u) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster_sync();  // every peer's barrier exists before anyone stores into it
    if (threadIdx.x == 0) {
        uint64_t state;
        const uint32_t bytes = (uint32_t)(N - 1) * npos * (uint32_t)kVecBytes;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                     : "=l"(state)
                     : "r"(my_bar), "r"(bytes)
                     : "memory");
    }
    // push: my slice into slot [r] of every peer (and of my own stage)
    const uint32_t slot_r = smem_u32(stage + (uint32_t)r * P);
#pragma unroll 1
    for (uint32_t v = threadIdx.x; v < npos; v += blockDim.x) {
        const uint4 x = (v == threadIdx.x) ? first : load_input<T>(p.send[r], pos0 + v, p.count);
        stage[(uint32_t)r * P + v] = x;
        if (drop == r) continue;
#pragma unroll 1
        for (int q = 0; q < N; ++q) {
            if (q == r) continue;
            st_async_v4(map_to_rank(slot_r + v * kVecBytes, (uint32_t)q), x, map_to_rank(my_bar, (uint32_t)q));
        }
    }
    // wait for the N-1 incoming slices (bounded)
    int ok = 1;
    {
        Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, r, 0);
        while (!mbar_try_wait(my_bar, 0u)) {
            if (waiter_expired(w)) {
                ok = 0;
                break;
            }
        }
    }
    if (ok) {
        // reduce in rank order; each thread reads its own stage[r] writes and
        // the peers' slots, which the mbarrier completion made visible
#pragma unroll 1
        for (uint32_t v = threadIdx.x; v < npos; v += blockDim.x) {
            typename M::Acc acc = M::load(stage[v]);
#pragma unroll 1
            for (int q = 1; q < N; ++q) M::add(acc, stage[(uint32_t)q * P + v]);
            store_output<T>(p.recv[r], pos0 + v, p.count, M::store(acc));
        }
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still store into its shared memory
    if (p.timing != nullptr && threadIdx.x == 0) {
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = globaltimer_ns();
    }
}

template <typename T>
static cudaError_t launch_cluster_t(const Params& p, int threads, size_t smem, cudaStream_t stream, bool pdl) {
    const void* k = (const void*)oneshot_cluster_kernel<T>;
    static bool configured[3] = {false, false, false};
    const int idx = sizeof(T) == 4 ? 0 : sizeof(T) == 2 ? 1 : 2;
    if (!configured[idx]) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kClusterStageBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[idx] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nranks * p.ctas_per_rank));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)p.nranks;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void* args[] = {(void*)&p};
    return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch_cluster(const Params& p, rra_dtype_t dtype, int threads, cudaStream_t stream, bool pdl) {
    const size_t smem = (size_t)p.nranks * p.per_cta * kVecBytes;
    if (smem > kClusterStageBytes || p.nranks > kClusterMaxRanks) return cudaErrorInvalidValue;
    switch (dtype) {
        case RRA_FP32: return launch_cluster_t<float>(p, threads, smem, stream, pdl);
        case RRA_BF16: return launch_cluster_t<__nv_bfloat16>(p, threads, smem, stream, pdl);
        case RRA_FP64: return launch_cluster_t<double>(p, threads, smem, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rra
