// fused.cu -- AllReduce with a residual-add epilogue, written on the public
// device-side API (include/rra_device.cuh).
//
// "Every Microsecond Matters" (Abstract; Sec. I, contributions; Fig. 6-9)
// provides a low-latency device API so that custom collective kernels can
// be built on it.  This is one such kernel: the AllReduce of a tensor-
// parallel layer together with the residual add that follows it,
//     recv[r] = round( sum_p x_p  +  res[r] ),
// the rank-order sum in the running type, the residual added to the running
// value, one rounding.  The partial sums never leave the SMs between the
// reduction and the add.
//
// One cluster of N CTAs per slice (CTA r = rank r), as the cluster
// AllReduce.  Two shapes, both on rra_dev::Team:
//   one-shot  every rank bcast()s its slice; every CTA reduces the slice and
//             adds its own residual (reads only its own rank's buffers);
//   two-shot  rank r send()s partition q of its slice to CTA q; CTA q reduces
//             partition q and, for every rank d, adds res[d] and stores into
//             recv[d] (outputs and residuals treated as registered symmetric
//             buffers, like the direct two-shot).
// A cluster handles slices c, c + G, c + 2G, ... of the message, one epoch
// each; with one slice per cluster (the default) that is a single epoch.
// With kBulk the pushes are the API's bulk sends (the TMA engine copies the
// slice, or each partition, from the input straight into the windows,
// the own slot included) instead of per-vector st.async sends.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "prims.cuh"
#include "rra_device.cuh"
#include "rra_internal.h"
#include "kernel_attrs.h"

namespace rra {

template <typename T, bool kTwoShot, bool kBulk>
__global__ void __launch_bounds__(256) residual_kernel(const __grid_constant__ FusedParams f) {
    using M = VecMath<T>;
    const Params& p = f.base;
    extern __shared__ __align__(16) uint4 window[];
    __shared__ __align__(8) uint64_t bars[2];
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t S = p.per_cta;
    const uint32_t Q = kTwoShot ? S / N : S;  // slot vectors
    const uint32_t G = (uint32_t)p.ctas_per_rank;
    const uint32_t nslices = p.nsteps;
    const uint32_t nt = blockDim.x;
    uint32_t cid;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cid));

    // positions of slice s, and how many of them this CTA reduces
    auto npos_of = [&](uint32_t s) { return min(S, p.nvec - s * S); };
    auto mine_of = [&](uint32_t s, uint32_t r) {
        const uint32_t np = npos_of(s);
        return kTwoShot ? (np > r * Q ? min(Q, np - r * Q) : 0u) : np;
    };

    // bytes a CTA receives per epoch: every peer's slot (and, with bulk
    // sends, its own)
    const uint32_t senders = kBulk ? N : N - 1;
    rra_dev::Team t;
    {
        uint32_t r0;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r0));
        t.setup(window, bars, Q, senders * mine_of(cid, r0) * (uint32_t)kVecBytes);
    }
    const uint32_t r = t.rank();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const uint64_t deadline = t_start + p.timeout_ns;
    const void* src = p.send[r];
    const uint32_t step = nt * (uint32_t)kClusterBatch;
    uint4 x[kClusterBatch];
    auto load_batch = [&](uint32_t base, uint32_t npos, uint32_t b0) {
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v < npos) x[j] = load_input<T>(src, base + v, p.count);
        }
    };
    // Residual vectors of this thread's first outputs of an epoch: one-shot,
    // its first kClusterBatch positions; two-shot, its first position for
    // the first kClusterBatch ranks.  Loaded early, consumed after the wait.
    uint4 rp[kClusterBatch];
    auto prefetch_residual = [&](uint32_t base, uint32_t mine) {
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            if (kTwoShot) {
                const uint32_t d = r + j < N ? r + j : r + j - N;
                if (threadIdx.x < mine && (uint32_t)j < N)
                    rp[j] = load_input<T>(f.resid[d], base + r * Q + threadIdx.x, p.count);
            } else {
                const uint32_t u = threadIdx.x + (uint32_t)j * nt;
                if (u < mine) rp[j] = load_input<T>(f.resid[r], base + u, p.count);
            }
        }
    };
    // the first epoch's first inputs and residuals are in flight while the
    // cluster barrier that guards the peers' windows completes
    if (!kBulk) load_batch(cid * S, npos_of(cid), 0);
    prefetch_residual(cid * S, mine_of(cid, r));
    const int32_t drop = p.drop_rank;
    const bool pushes = drop != (int32_t)r;
    uint64_t* const tr = (p.trace != nullptr && threadIdx.x == 0) ? p.trace + (uint64_t)blockIdx.x * kTracePoints
                                                                   : nullptr;
    if (tr) {
        tr[0] = t_start;
        tr[1] = globaltimer_after((kBulk ? 0ull : (uint64_t)x[0].x) + (uint64_t)(uint32_t)drop);
    }
    t.ready();
    if (tr) tr[2] = globaltimer_ns();

    uint32_t k = 0;
    bool arrived = false;  // t.sent() done (CTA-uniform)
#pragma unroll 1
    for (uint32_t s = cid; s < nslices; s += G, ++k) {
        if (k > 0) t.advance_epoch(senders * mine_of(s, r) * (uint32_t)kVecBytes);
        const uint32_t base = s * S;
        const uint32_t npos = npos_of(s);
        const uint32_t mine = mine_of(s, r);
        if (kBulk) {
            // whole runs of vectors straight from the input into the windows
            const char* const in = (const char*)src + (size_t)base * kVecBytes;
            if (kTwoShot) {
                const uint32_t q = threadIdx.x;  // partition q to CTA q
                const uint32_t len = q < N && npos > q * Q ? min(Q, npos - q * Q) : 0u;
                if (len != 0 && (q == r || pushes)) t.bulk_send(q, 0, in + (size_t)q * Q * kVecBytes, len);
            } else if (threadIdx.x == 0) {
                t.bulk_bcast(0, in, npos, pushes ? (1u << N) - 1u : 1u << r);
            }
        }
        // exchange, one batch of input loads in flight per thread
#pragma unroll 1
        for (uint32_t b0 = 0; !kBulk && b0 < npos; b0 += step) {
            if (k > 0 || b0 > 0) load_batch(base, npos, b0);
#pragma unroll
            for (int j = 0; j < kClusterBatch; ++j) {
                const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
                if (v >= npos) continue;
                if (kTwoShot) {
                    const uint32_t q = v / Q;
                    const uint32_t u = v - q * Q;
                    if (q == r) t.put(u, x[j]);
                    else if (pushes) t.send(q, u, x[j]);
                } else {
                    if (pushes) t.bcast(v, x[j]);
                    t.put(v, x[j]);
                }
            }
        }
        if (tr && k == 0) tr[3] = globaltimer_ns();
        if (!kBulk && s + G >= nslices) {  // that was this CTA's last send: start the exit barrier now
            t.sent();
            arrived = true;
        }
        if (k > 0) prefetch_residual(base, mine);
        if (!t.wait(deadline)) {
            if (threadIdx.x == 0) record_error(p.ctrl, RRA_ERR_TIMEOUT, (int)r, (int)k);
            break;
        }
        if (tr && k == 0) tr[4] = globaltimer_ns();
        // reduce in rank order, add the residual to the running value, round once
        auto sum_at = [&](uint32_t u) {
            typename M::Acc acc = M::load(t.recv(0, u));
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, t.recv(q, u));
            return acc;
        };
        if (kTwoShot) {
#pragma unroll 1
            for (uint32_t u = threadIdx.x; u < mine; u += nt) {
                const typename M::Acc acc = sum_at(u);
                const uint32_t pos = base + r * Q + u;
                const bool first = u == threadIdx.x;  // its residuals were prefetched
#pragma unroll
                for (uint32_t d0 = 0; d0 < (uint32_t)kClusterMaxRanks; ++d0) {
                    if (d0 >= N) break;
                    const uint32_t d = r + d0 < N ? r + d0 : r + d0 - N;
                    typename M::Acc out = acc;
                    M::add(out, first && d0 < (uint32_t)kClusterBatch ? rp[d0 % kClusterBatch]
                                                                      : load_input<T>(f.resid[d], pos, p.count));
                    store_output<T>(p.recv[d], pos, p.count, M::store(out));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < kClusterBatch; ++j) {
                const uint32_t u = threadIdx.x + (uint32_t)j * nt;
                if (u < mine) {
                    typename M::Acc acc = sum_at(u);
                    M::add(acc, rp[j]);
                    store_output<T>(p.recv[r], base + u, p.count, M::store(acc));
                }
            }
#pragma unroll 1
            for (uint32_t u = threadIdx.x + (uint32_t)kClusterBatch * nt; u < mine; u += nt) {
                typename M::Acc acc = sum_at(u);
                M::add(acc, load_input<T>(f.resid[r], base + u, p.count));
                store_output<T>(p.recv[r], base + u, p.count, M::store(acc));
            }
        }
    }
    if (!arrived) t.sent();  // left the loop early (a wait ran out)
    t.finish();
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
    if (tr) tr[5] = globaltimer_ns();
}

template <typename T>
static const void* residual_kernel_for(bool two_shot, bool bulk) {
    if (bulk) return two_shot ? (const void*)residual_kernel<T, true, true> : (const void*)residual_kernel<T, false, true>;
    return two_shot ? (const void*)residual_kernel<T, true, false> : (const void*)residual_kernel<T, false, false>;
}

static const void* residual_kernel_ptr(rra_dtype_t dtype, bool two_shot, bool bulk) {
    switch (dtype) {
        case RRA_FP32: return residual_kernel_for<float>(two_shot, bulk);
        case RRA_BF16: return residual_kernel_for<__nv_bfloat16>(two_shot, bulk);
        case RRA_FP64: return residual_kernel_for<double>(two_shot, bulk);
    }
    return nullptr;
}

static cudaError_t configure_residual(const void* k) { return configure_cluster_kernel(k, (int)kClusterStageBytes); }

size_t residual_stage_bytes(const Params& p, bool two_shot) {
    const size_t q = two_shot ? p.per_cta / (uint32_t)p.nranks : p.per_cta;
    return 2 * (size_t)p.nranks * q * kVecBytes;  // two sub-buffers
}

cudaError_t launch_residual(const FusedParams& f, rra_dtype_t dtype, bool two_shot, bool bulk, int threads,
                            cudaStream_t stream, bool pdl) {
    const Params& p = f.base;
    const size_t smem = residual_stage_bytes(p, two_shot);
    if (smem == 0 || smem > kClusterStageBytes || p.nranks < 2 || p.nranks > kClusterMaxRanks)
        return cudaErrorInvalidValue;
    if (two_shot && p.per_cta % (uint32_t)p.nranks != 0) return cudaErrorInvalidValue;
    if (bulk && two_shot && threads < p.nranks) return cudaErrorInvalidValue;  // threads 0..N-1 issue the copies
    const void* k = residual_kernel_ptr(dtype, two_shot, bulk);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = configure_residual(k);
    if (e != cudaSuccess) return e;
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
    void* args[] = {(void*)&f};
    return cudaLaunchKernelExC(&cfg, k, args);
}

int residual_max_active(rra_dtype_t dtype, bool two_shot, bool bulk, int nranks, int threads, size_t smem) {
    const void* k = residual_kernel_ptr(dtype, two_shot, bulk);
    if (k == nullptr || configure_residual(k) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nranks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)nranks;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rra
