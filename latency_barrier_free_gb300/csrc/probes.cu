// probes.cu -- single-GPU latency-floor probes (include/rra_probe.h).
//
// "Every Microsecond Matters", Sec. VI: L_SoL = 2 * L_L2_RTT + L_remote_store.
// L_L2_RTT is measured here as the per-hop time of a dependent pointer chase
// through an L2-resident buffer (the review of the paper points out that a
// fence's latency is not a load-to-use time); L_remote_store as half the
// round trip of a fence-free store/poll ping-pong between two SMs.
// The same model for the transport of the cluster kernels: a bulk copy from
// an L2-resident input straight into a peer CTA's shared memory, whose
// arrival completes the peer's mbarrier (half the round trip of a bulk-copy
// ping-pong inside one cluster), plus the one cluster barrier such a kernel
// must pass before its first push.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <numeric>
#include <random>
#include <vector>

#include "cluster_prims.cuh"
#include "rra.h"
#include "rra_probe.h"

namespace {

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

// out[0] = elapsed ns of the timed pass, out[1] = final index (keeps the chain live)
__global__ void chase_kernel(const uint64_t* next, uint64_t nwords, uint64_t hops, uint64_t* out) {
    uint64_t i = 0;
    for (uint64_t h = 0; h < nwords; ++h) i = ld_cg_u64(next + i);  // warm pass: whole cycle into L2
    const uint64_t t0 = gtimer();
    for (uint64_t h = 0; h < hops; ++h) i = ld_cg_u64(next + i);
    const uint64_t t1 = gtimer();
    out[0] = t1 - t0;
    out[1] = i;
}

// flags[0]: a -> b, flags[32]: b -> a (separate 128-byte lines).
// res[0] = round trips ns total, res[1] = smid a, res[2] = smid b, res[3] = error
__global__ void pingpong_kernel(uint32_t* flags, int cta_a, int cta_b, int warm, int iters, uint64_t* res) {
    if (threadIdx.x != 0) return;
    const int me = (int)blockIdx.x;
    if (me != cta_a && me != cta_b) return;
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const uint64_t deadline = gtimer() + 1000000000ull;  // 1 s
    uint32_t* to_b = flags;
    uint32_t* to_a = flags + 32;
    const int total = warm + iters;
    if (me == cta_a) {
        res[1] = smid;
        uint64_t t0 = 0;
        for (int i = 1; i <= total; ++i) {
            if (i == warm + 1) t0 = gtimer();
            st_relaxed(to_b, (uint32_t)i);
            uint32_t spins = 0;
            while (ld_relaxed(to_a) != (uint32_t)i) {
                if ((++spins & 255u) == 0u && gtimer() > deadline) { res[3] = 1; return; }
            }
        }
        res[0] = gtimer() - t0;
    } else {
        res[2] = smid;
        for (int i = 1; i <= total; ++i) {
            uint32_t spins = 0;
            while (ld_relaxed(to_b) != (uint32_t)i) {
                if ((++spins & 255u) == 0u && gtimer() > deadline) { res[3] = 1; return; }
            }
            st_relaxed(to_a, (uint32_t)i);
        }
    }
}

// Bulk-copy ping-pong between the two CTAs of a cluster.  CTA 0 copies 128
// bytes from `src` (global memory, L2-resident after the first round) into
// CTA 1's shared memory with one bulk copy that completes CTA 1's mbarrier;
// CTA 1's wait returns and it answers the same way into CTA 0; CTA 0's wait
// returns.  Then both run `iters` cluster barriers (relaxed arrive + acquire
// wait, as the cluster kernels use them).  Every wait is bounded (1 s).
// res[0] = ns of `iters` round trips after `warm`, res[1] = ns of `iters`
// cluster barriers (CTA 0), res[2] = error flag, res[3], res[4] = SM ids.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32)
    dsmem_pingpong_kernel(const uint4* src, int warm, int iters, uint64_t* res) {
    __shared__ __align__(128) uint4 buf[8];
    __shared__ __align__(8) uint64_t bar;
    const uint32_t me = rra::cluster_ctarank();
    const uint32_t peer = me ^ 1u;
    const uint32_t bar_s = rra::smem_u32(&bar);
    const uint32_t buf_s = rra::smem_u32(buf);
    if (threadIdx.x == 0) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        res[3 + me] = smid;
        rra::mbar_init(bar_s, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        rra::mbar_expect_tx(bar_s, 128u);  // the arrival of phase 0
    }
    __syncwarp();
    rra::cluster_sync();  // both mbarriers exist
    const uint64_t deadline = gtimer() + 1000000000ull;
    int ok = 1;
    uint32_t parity = 0;
    uint64_t t0 = 0;
    auto wait_own = [&]() {
        uint32_t spins = 0;
        while (!rra::mbar_try_wait(bar_s, parity)) {
            if ((++spins & 63u) == 0u && gtimer() > deadline) return false;
        }
        return true;
    };
    for (int i = 0; i < warm + iters && ok; ++i) {
        if (me == 0 && i == warm) t0 = gtimer();
        if (me == 0) {
            if (threadIdx.x == 0) rra::bulk_g2s_multicast(buf_s, src, 128u, bar_s, (uint16_t)(1u << peer));
            ok = __all_sync(0xffffffffu, wait_own());  // warp-uniform: the cluster barriers below are .aligned
            if (ok && threadIdx.x == 0) rra::mbar_expect_tx(bar_s, 128u);  // the arrival of the next phase
        } else {
            ok = __all_sync(0xffffffffu, wait_own());
            if (ok && threadIdx.x == 0) {
                rra::mbar_expect_tx(bar_s, 128u);
                rra::bulk_g2s_multicast(buf_s, src, 128u, bar_s, (uint16_t)(1u << peer));
            }
        }
        parity ^= 1u;
    }
    if (me == 0 && threadIdx.x == 0) res[0] = ok ? gtimer() - t0 : 0ull;
    if (!ok && threadIdx.x == 0) res[2] = 1ull;
    const uint64_t t1 = gtimer();
    for (int i = 0; i < iters; ++i) {
        rra::cluster_arrive_relaxed();
        rra::cluster_wait();
    }
    if (me == 0 && threadIdx.x == 0) res[1] = gtimer() - t1;
    rra::cluster_sync();  // no CTA leaves while a copy into the other may be in flight
}

__global__ void empty_kernel() {}

struct BigParams {
    uint64_t words[144];  // 1152 bytes, the size of the AllReduce parameter block
};
// The launch copies the parameter block whether or not the body reads it.
__global__ void empty_kernel_big(const __grid_constant__ BigParams p) { (void)p; }

// An empty kernel shaped like the AllReduce kernels' launches: it releases
// the next kernel and waits for the previous one as they do (programmatic
// dependent launch), and does nothing else.
__global__ void chain_kernel() {
    rra::pdl_release_early();
    rra::pdl_wait();
}

// Host-link probes: threads stream 16-byte vectors, grid-strided, through
// pinned host memory mapped into the device's address space (the reads with
// kLinkBatch loads in flight per thread).  The read folds the vectors into
// one word that is stored only if it matches a value no input has (so the
// loads stay live).
constexpr int kLinkBatch = 4;

__global__ void link_read_kernel(const uint4* __restrict__ src, size_t n, uint4* sink) {
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += stride * kLinkBatch) {
        uint4 v[kLinkBatch];
#pragma unroll
        for (int k = 0; k < kLinkBatch; ++k) {
            const size_t i = i0 + (size_t)k * stride;
            v[k] = i < n ? src[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kLinkBatch; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    if (acc == 0xFFFFFFFFu) sink[0] = make_uint4(acc, 0u, 0u, 0u);
}

__global__ void link_write_kernel(uint4* dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = make_uint4((uint32_t)i, 0u, 0u, 0u);
}

__global__ void link_copy_kernel(const uint4* __restrict__ src, uint4* dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

}  // namespace

extern "C" {

rra_status_t rra_probe_sm_count(int* sms) {
    if (sms == nullptr) return RRA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RRA_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return RRA_ERR_CUDA;
    return RRA_OK;
}

rra_status_t rra_probe_l2_chase(size_t buf_bytes, uint64_t hops, uint64_t seed, double* ns_per_hop) {
    if (ns_per_hop == nullptr || buf_bytes < (64u << 10) || hops == 0 || buf_bytes > (1ull << 31))
        return RRA_ERR_INVALID_ARG;
    const uint64_t n = buf_bytes / 8;
    // One random cycle through all words: Sattolo's algorithm.
    std::vector<uint64_t> perm(n);
    std::iota(perm.begin(), perm.end(), 0ull);
    std::mt19937_64 g(seed);
    for (uint64_t i = n - 1; i > 0; --i) {
        std::uniform_int_distribution<uint64_t> d(0, i - 1);
        std::swap(perm[i], perm[d(g)]);
    }
    std::vector<uint64_t> next(n);
    for (uint64_t i = 0; i < n; ++i) next[perm[i]] = perm[(i + 1) % n];
    uint64_t* dnext = nullptr;
    uint64_t* dout = nullptr;
    if (cudaMalloc((void**)&dnext, n * 8) != cudaSuccess) { cudaGetLastError(); return RRA_ERR_OOM; }
    if (cudaMalloc((void**)&dout, 16) != cudaSuccess) { cudaGetLastError(); cudaFree(dnext); return RRA_ERR_OOM; }
    rra_status_t st = RRA_OK;
    uint64_t out[2] = {0, 0};
    if (cudaMemcpy(dnext, next.data(), n * 8, cudaMemcpyHostToDevice) != cudaSuccess) st = RRA_ERR_CUDA;
    if (st == RRA_OK) {
        chase_kernel<<<1, 1>>>(dnext, n, hops, dout);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(out, dout, 16, cudaMemcpyDeviceToHost) != cudaSuccess)
            st = RRA_ERR_CUDA;
    }
    cudaFree(dnext);
    cudaFree(dout);
    if (st == RRA_OK) *ns_per_hop = (double)out[0] / (double)hops;
    return st;
}

rra_status_t rra_probe_pingpong(int cta_a, int cta_b, int iters, double* ns_round_trip, int* sm_a, int* sm_b) {
    if (ns_round_trip == nullptr || iters <= 0 || iters > (1 << 24) || cta_a == cta_b || cta_a < 0 || cta_b < 0)
        return RRA_ERR_INVALID_ARG;
    int dev = 0, sms = 0, smem_max = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
        return RRA_ERR_CUDA;
    if (cta_a >= sms || cta_b >= sms || !coop) return RRA_ERR_INVALID_ARG;
    // One CTA per SM: each CTA asks for more than half of the SM's shared memory.
    const int smem = smem_max;
    if (cudaFuncSetAttribute(pingpong_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return RRA_ERR_CUDA;
    uint32_t* flags = nullptr;
    uint64_t* res = nullptr;
    if (cudaMalloc((void**)&flags, 256) != cudaSuccess) { cudaGetLastError(); return RRA_ERR_OOM; }
    if (cudaMalloc((void**)&res, 32) != cudaSuccess) { cudaGetLastError(); cudaFree(flags); return RRA_ERR_OOM; }
    rra_status_t st = RRA_OK;
    uint64_t h[4] = {0, 0, 0, 0};
    if (cudaMemset(flags, 0, 256) != cudaSuccess || cudaMemset(res, 0, 32) != cudaSuccess) st = RRA_ERR_CUDA;
    if (st == RRA_OK) {
        int warm = std::max(1, iters / 8);
        void* args[] = {(void*)&flags, (void*)&cta_a, (void*)&cta_b, (void*)&warm, (void*)&iters, (void*)&res};
        if (cudaLaunchCooperativeKernel((const void*)pingpong_kernel, dim3(sms), dim3(32), args, (size_t)smem, 0) !=
                cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(h, res, 32, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            st = RRA_ERR_CUDA;
        }
    }
    cudaFree(flags);
    cudaFree(res);
    if (st != RRA_OK) return st;
    if (h[3] != 0) return RRA_ERR_TIMEOUT;
    *ns_round_trip = (double)h[0] / (double)iters;
    if (sm_a) *sm_a = (int)h[1];
    if (sm_b) *sm_b = (int)h[2];
    return RRA_OK;
}

rra_status_t rra_probe_dsmem_pingpong(int iters, double* ns_round_trip, double* ns_cluster_barrier, int* sm_a,
                                      int* sm_b) {
    if (ns_round_trip == nullptr || ns_cluster_barrier == nullptr || iters <= 0 || iters > (1 << 22))
        return RRA_ERR_INVALID_ARG;
    uint4* src = nullptr;
    uint64_t* res = nullptr;
    if (cudaMalloc((void**)&src, 128) != cudaSuccess) { cudaGetLastError(); return RRA_ERR_OOM; }
    if (cudaMalloc((void**)&res, 64) != cudaSuccess) { cudaGetLastError(); cudaFree(src); return RRA_ERR_OOM; }
    rra_status_t st = RRA_OK;
    uint64_t h[8] = {};
    if (cudaMemset(src, 0, 128) != cudaSuccess || cudaMemset(res, 0, 64) != cudaSuccess) st = RRA_ERR_CUDA;
    if (st == RRA_OK) {
        const int warm = std::max(1, iters / 8);
        dsmem_pingpong_kernel<<<2, 32>>>(src, warm, iters, res);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(h, res, 64, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            st = RRA_ERR_CUDA;
        }
    }
    cudaFree(src);
    cudaFree(res);
    if (st != RRA_OK) return st;
    if (h[2] != 0) return RRA_ERR_TIMEOUT;
    *ns_round_trip = (double)h[0] / (double)iters;
    *ns_cluster_barrier = (double)h[1] / (double)iters;
    if (sm_a) *sm_a = (int)h[3];
    if (sm_b) *sm_b = (int)h[4];
    return RRA_OK;
}

rra_status_t rra_probe_empty_kernel(rra_stream_t stream) {
    empty_kernel<<<1, 32, 0, (cudaStream_t)stream>>>();
    return cudaGetLastError() == cudaSuccess ? RRA_OK : RRA_ERR_CUDA;
}

rra_status_t rra_probe_launch_shape(int ctas, int threads, int big_params, int cooperative, rra_stream_t stream) {
    if (ctas < 1 || ctas > 4096 || threads < 32 || threads > 1024) return RRA_ERR_INVALID_ARG;
    static BigParams bp = {};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 1 : 0;
    cudaError_t e;
    if (big_params) {
        void* args[] = {(void*)&bp};
        e = cudaLaunchKernelExC(&cfg, (const void*)empty_kernel_big, args);
    } else {
        e = cudaLaunchKernelExC(&cfg, (const void*)empty_kernel, nullptr);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    return RRA_OK;
}

rra_status_t rra_probe_launch_chain(int ctas, int threads, int cluster, int pdl, rra_stream_t stream) {
    if (ctas < 1 || ctas > 4096 || threads < 32 || threads > 1024 || cluster < 1 || cluster > 8 ||
        ctas % cluster != 0)
        return RRA_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelExC(&cfg, (const void*)chain_kernel, nullptr) != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    return RRA_OK;
}

rra_status_t rra_probe_host_link(size_t bytes, int iters, double* read_gbps, double* write_gbps,
                                 double* copy_gbps) {
    if (read_gbps == nullptr || write_gbps == nullptr || copy_gbps == nullptr || bytes < (64u << 10) ||
        bytes > (1ull << 30) || bytes % 16 != 0 || iters <= 0 || iters > 10000)
        return RRA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return RRA_ERR_CUDA;
    uint4 *h_src = nullptr, *h_dst = nullptr, *m_src = nullptr, *m_dst = nullptr, *sink = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    rra_status_t st = RRA_OK;
    if (cudaHostAlloc((void**)&h_src, bytes, cudaHostAllocMapped) != cudaSuccess ||
        cudaHostAlloc((void**)&h_dst, bytes, cudaHostAllocMapped) != cudaSuccess ||
        cudaMalloc((void**)&sink, 16) != cudaSuccess) {
        cudaGetLastError();
        st = RRA_ERR_OOM;
    }
    if (st == RRA_OK && (cudaHostGetDevicePointer((void**)&m_src, h_src, 0) != cudaSuccess ||
                         cudaHostGetDevicePointer((void**)&m_dst, h_dst, 0) != cudaSuccess ||
                         cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)) {
        cudaGetLastError();
        st = RRA_ERR_CUDA;
    }
    const size_t n = bytes / 16;
    if (st == RRA_OK) {
        for (size_t i = 0; i < n; ++i) h_src[i] = make_uint4((uint32_t)i, 1u, 2u, 3u);
    }
    // mean of `iters` launches after two warm-ups.  Read and write: two CTAs
    // of 256 threads per SM.  Copy: one CTA of 128 threads per SM, one vector
    // in flight per thread, so that every thread's next load overlaps other
    // threads' stores (with all of a small buffer in flight at once, the
    // reads and the writes would run one after the other)
    const dim3 grid((unsigned)(2 * sms)), block(256), cgrid((unsigned)sms), cblock(128);
    auto measure = [&](int which, double* gbps) {
        if (st != RRA_OK) return;
        for (int r = -2; r < iters; ++r) {
            if (r == 0 && cudaEventRecord(e0) != cudaSuccess) break;
            if (which == 0) link_read_kernel<<<grid, block>>>(m_src, n, sink);
            else if (which == 1) link_write_kernel<<<grid, block>>>(m_dst, n);
            else link_copy_kernel<<<cgrid, cblock>>>(m_src, m_dst, n);
        }
        float ms = 0.f;
        if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e1) != cudaSuccess ||
            cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.f) {
            cudaGetLastError();
            st = RRA_ERR_CUDA;
            return;
        }
        *gbps = (double)bytes * iters / ((double)ms * 1e6);
    };
    measure(0, read_gbps);
    measure(1, write_gbps);
    measure(2, copy_gbps);
    if (st == RRA_OK && cudaDeviceSynchronize() != cudaSuccess) st = RRA_ERR_CUDA;
    if (st == RRA_OK && std::memcmp(h_src, h_dst, bytes) != 0) st = RRA_ERR_CUDA;  // the copy arrived whole
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (sink) cudaFree(sink);
    if (h_src) cudaFreeHost(h_src);
    if (h_dst) cudaFreeHost(h_dst);
    return st;
}

}  // extern "C"
