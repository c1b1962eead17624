// cluster.cu -- push AllReduce through distributed shared memory.
//
// "Every Microsecond Matters", Sec. III-A (one-shot and two-shot, push) and
// Sec. IV (data arrival as the only synchronisation), restated for what one
// GB300 offers below L2: the CTAs of a thread-block cluster sit on one GPC,
// are scheduled together by the hardware, and can store into each other's
// shared memory.  A cluster holds one CTA per virtual rank for one slice of
// the message; CTA r's shared memory is rank r's window for that slice.  A
// CTA reads only its own rank's input and writes only into peers' windows
// (and, for the two-shot, into every rank's output).  A push is an st.async
// (cluster_kernel), or a TMA bulk copy straight from the rank's input
// (cluster_tma_kernel, multicast to all N CTAs for the one-shot); either
// completes the receiver's mbarrier transaction count: the receiver waits on
// its own mbarrier -- the arrival of the bytes is the signal -- and adds the
// N contributions in rank order (bit-identical to the other fixed-order
// kernels).
//
//   one-shot: rank r pushes its whole slice into slot [r] of every peer; each
//             CTA reduces the slice and stores it into its own rank's output.
//   two-shot: the slice is cut into N partitions; rank r pushes partition q
//             into slot [r] of CTA q only (the ReduceScatter), CTA q reduces
//             partition q and stores it into every rank's output (the
//             AllGather, as direct stores into the outputs, which are treated
//             as registered symmetric buffers, Sec. II-B).  N times less
//             shared-memory traffic and stage than the one-shot, the same
//             single synchronisation hop, and HBM sees only the compulsory
//             N*M bytes read and N*M written.
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

#include "cluster_prims.cuh"
#include "prims.cuh"
#include "rra_internal.h"
#include "kernel_attrs.h"

namespace rra {

// One slice per cluster, CTA r of the cluster = rank r.  Stage layout: N
// slots of Q vectors, slot [q] = rank q's contribution; Q = S (one-shot) or
// S / N (two-shot), S = p.per_cta vectors per slice.  kTrace: the variant
// with trace points (rra_comm_set_trace), launched only while a trace buffer
// is set; the untraced kernel is smaller, and calls measured about 4 %
// shorter on it (N = 4, 128 B-1 MiB, graph replay).
template <typename T, bool kTwoShot, bool kTrace>
__global__ void __launch_bounds__(256) cluster_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t Q = kTwoShot ? S / N : S;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const void* src = p.send[r];
    // positions this CTA reduces: the whole slice, or partition r of it
    const uint32_t mine = kTwoShot ? (npos > r * Q ? min(Q, npos - r * Q) : 0u) : npos;

    // The barrier lives in this launch's shared memory, so it is set up
    // before waiting for the previous kernel; its phase completes when the
    // N-1 contributions' bytes have arrived.  The cluster barrier that makes
    // it visible to the peers is split: arrive now, wait just before the
    // first push, so its latency overlaps the input loads.  The arrive is
    // relaxed: fence.mbarrier_init already orders the initialisation before
    // it, and a release would stall every thread on a memory barrier.
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, (N - 1) * mine * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();

    // first batch of inputs and the injected-fault word, in flight together
    uint4 x[kClusterBatch];
#pragma unroll
    for (int j = 0; j < kClusterBatch; ++j) {
        const uint32_t v = threadIdx.x + (uint32_t)j * nt;
        x[j] = make_uint4(0, 0, 0, 0);
        if (v < npos) x[j] = load_input<T>(src, base + v, p.count);
    }
    const int32_t drop = p.drop_rank;
    uint64_t* const tr = (kTrace && p.trace != nullptr && threadIdx.x == 0)
                             ? p.trace + (uint64_t)blockIdx.x * kTracePoints
                             : nullptr;
    if (tr) {
        tr[0] = t_start;
        tr[1] = globaltimer_after((uint64_t)x[0].x + (uint64_t)(uint32_t)drop);
    }
    cluster_wait();  // every peer's barrier exists before anyone stores into it
    if (tr) tr[2] = globaltimer_ns();

    // push: vector v of my slice goes to slot [r] of its destination(s)
    const uint32_t slot_r = smem_u32(stage + r * Q);
    const uint32_t step = nt * (uint32_t)kClusterBatch;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < npos; b0 += step) {
        if (b0 != 0) {
#pragma unroll
            for (int j = 0; j < kClusterBatch; ++j) {
                const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
                if (v < npos) x[j] = load_input<T>(src, base + v, p.count);
            }
        }
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v >= npos) continue;
            if (kTwoShot) {
                const uint32_t q = v / Q;
                const uint32_t u = v - q * Q;
                if (q == r) {
                    stage[r * Q + u] = x[j];
                } else if (drop != (int32_t)r) {
                    st_async_v4(map_to_rank(slot_r + u * (uint32_t)kVecBytes, q), x[j], map_to_rank(my_bar, q));
                }
            } else {
                if (drop != (int32_t)r) {
#pragma unroll 1
                    for (uint32_t k = 1; k < N; ++k) {
                        const uint32_t q = r + k < N ? r + k : r + k - N;
                        st_async_v4(map_to_rank(slot_r + v * (uint32_t)kVecBytes, q), x[j], map_to_rank(my_bar, q));
                    }
                }
                stage[r * Q + v] = x[j];
            }
        }
    }
    // Second cluster barrier, split and relaxed: arriving says "my pushes are
    // issued".  It orders no data (a release here would stall until the
    // pushes are acknowledged).  A CTA leaves only after its own mbarrier has
    // seen every incoming byte, or, if its wait ran out, after every peer
    // has issued its pushes (at least a poll time limit ago).
    cluster_arrive_relaxed();
    if (tr) tr[3] = globaltimer_ns();
    // wait for the N-1 incoming contributions (bounded)
    int ok = 1;
    {
        Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, (int)r, 0);
        while (!mbar_try_wait(my_bar, 0u)) {
            if (waiter_expired(w)) {
                ok = 0;
                break;
            }
        }
    }
    if (tr && ok) tr[4] = globaltimer_ns();
    if (kTwoShot) __syncthreads();  // my own slot was written by other threads of this CTA
    if (ok) {
        // reduce in rank order; the mbarrier completion made the peers' slots visible
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * Q + u]);
            const uint4 out = M::store(acc);
            if (kTwoShot) {
                const uint32_t pos = base + r * Q + u;
#pragma unroll 1
                for (uint32_t k = 0; k < N; ++k) {
                    const uint32_t d = r + k < N ? r + k : r + k - N;
                    store_output<T>(p.recv[d], pos, p.count, out);
                }
            } else {
                store_output<T>(p.recv[r], base + u, p.count, out);
            }
        }
    }
    // A thread whose wait ran out keeps the CTA's shared memory alive until
    // every peer has issued its pushes into it.  After a completed wait every
    // incoming byte has landed and no peer will touch this memory again, so
    // the thread leaves without waiting (exited threads count as arrived).
    if (!__all_sync(0xffffffffu, ok)) cluster_wait();  // warp-uniform, as .aligned requires
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
    if (tr) tr[5] = globaltimer_ns();
}

// The same one-shot / two-shot with the push made by the TMA engine: a
// rank's CTA issues bulk copies from its own input straight into the
// peers' windows (one multicast copy of the slice to all N CTAs for the
// one-shot; one copy of partition q to CTA q for the two-shot), each
// completing the destination's mbarrier; no data passes through registers
// on the way out.  A copy covers whole 16-byte vectors: the last vector of
// an input whose size is not a multiple of 16 bytes is read in full (it
// lies in the same 16-byte block as valid data, so in the same page), and
// its extra lanes are never stored.  Since a CTA cannot see when its own
// copies into peers have landed, it leaves only after a cluster barrier
// that every CTA arrives at once its own incoming bytes are in.  kTrace: as
// for cluster_kernel.  kResidual (one-shot only): the fused AllReduce +
// residual add, every output round(rank-order sum + that rank's residual),
// the residual added to the running value, one rounding.  (A two-shot form,
// whose partition owners add every destination's residual, measured slower
// than the device-API kernel of fused.cu at two-shot sizes.)
template <typename T, bool kTwoShot, bool kTrace, bool kResidual>
__device__ __forceinline__ void tma_body(const Params& p, const void* const* resid) {
    static_assert(!(kTwoShot && kResidual), "the residual epilogue is the one-shot's");
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t Q = kTwoShot ? S / N : S;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const char* const src = (const char*)p.send[r];
    const uint32_t mine = kTwoShot ? (npos > r * Q ? min(Q, npos - r * Q) : 0u) : npos;

    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, N * mine * (uint32_t)kVecBytes);  // every slot, the own one included
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    uint64_t* const tr = (kTrace && p.trace != nullptr && threadIdx.x == 0)
                             ? p.trace + (uint64_t)blockIdx.x * kTracePoints
                             : nullptr;
    if (tr) {
        tr[0] = t_start;
        tr[1] = globaltimer_after((uint64_t)(uint32_t)drop);
    }
    // the residual of this thread's first output, read while the copies fly
    uint4 rv0 = make_uint4(0u, 0u, 0u, 0u);
    if (kResidual && threadIdx.x < mine) rv0 = load_input<T>(resid[r], base + threadIdx.x, p.count);
    cluster_wait();  // every peer's barrier exists before any copy completes on it
    if (tr) tr[2] = globaltimer_ns();
    const bool pushes = drop != (int32_t)r;
    if (kTwoShot) {
        // thread q: partition q of my slice into slot [r] of CTA q
        const uint32_t q = threadIdx.x;
        const uint32_t len = q < N && npos > q * Q ? min(Q, npos - q * Q) : 0u;
        if (len != 0 && (q == r || pushes))
            bulk_g2s_multicast(smem_u32(stage + r * Q), src + (size_t)(base + q * Q) * kVecBytes,
                               len * (uint32_t)kVecBytes, my_bar, (uint16_t)(1u << q));
    } else if (threadIdx.x == 0) {
        const uint16_t all = (uint16_t)((1u << N) - 1u);
        bulk_g2s_multicast(smem_u32(stage + r * Q), src + (size_t)base * kVecBytes, npos * (uint32_t)kVecBytes,
                           my_bar, pushes ? all : (uint16_t)(1u << r));
    }
    if (tr) tr[3] = globaltimer_ns();
    int ok = 1;
    {
        Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, (int)r, 0);
        while (!mbar_try_wait(my_bar, 0u)) {
            if (waiter_expired(w)) {
                ok = 0;
                break;
            }
        }
    }
    if (tr && ok) tr[4] = globaltimer_ns();
    cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    if (ok) {
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * Q + u]);
            const uint4 out = M::store(acc);
            if (kTwoShot) {
                const uint32_t pos = base + r * Q + u;
#pragma unroll 1
                for (uint32_t k = 0; k < N; ++k) {
                    const uint32_t d = r + k < N ? r + k : r + k - N;
                    store_output<T>(p.recv[d], pos, p.count, out);
                }
            } else if (kResidual) {
                M::add(acc, u == threadIdx.x ? rv0 : load_input<T>(resid[r], base + u, p.count));
                store_output<T>(p.recv[r], base + u, p.count, M::store(acc));
            } else {
                store_output<T>(p.recv[r], base + u, p.count, out);
            }
        }
    }
    cluster_wait();  // every CTA's incoming bytes are in: none of my copies is still in flight
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
    if (tr) tr[5] = globaltimer_ns();
}

template <typename T, bool kTwoShot, bool kTrace>
__global__ void __launch_bounds__(256) cluster_tma_kernel(const __grid_constant__ Params p) {
    tma_body<T, kTwoShot, kTrace, false>(p, nullptr);
}

template <typename T, bool kTrace>
__global__ void __launch_bounds__(256) cluster_tma_residual_kernel(const __grid_constant__ FusedParams f) {
    tma_body<T, false, kTrace, true>(f.base, f.resid);
}

// More ranks than CTAs in a cluster (N > 16): CTA j of a cluster of G = 16
// CTAs hosts ranks j, j + G, j + 2G, ... (< N), reading each hosted rank's
// input and writing each hosted rank's output.  A window holds a slot per
// rank; a push goes to the G - 1 other CTAs (every rank they host sees the
// same window), and the reduction still adds all N slots in rank order.
//   one-shot: each CTA receives every other rank's slice and reduces it;
//   two-shot: the slice is cut into G parts, CTA q reduces part q over all N
//             ranks and stores it into every rank's output (direct).
//
// With kResidual (the fused AllReduce + residual add above 16 ranks), every
// output is round(rank-order sum + that rank's residual), the residual added
// to the running value as by the one-cluster fused kernel.
//
// With kBulk the pushes are TMA bulk copies straight from the hosted ranks'
// inputs (device memory of this GPU, checked by the host): one-shot, thread
// m copies hosted rank m's slice into its slot of every CTA with cluster
// multicast; two-shot, thread (m, q) copies partition q of hosted rank m's
// slice into its slot of CTA q.  Every slot then arrives by copy, the own
// CTA's included, and a CTA leaves only after a cluster barrier that every
// CTA reaches once its own incoming bytes are in, so that no copy it issued
// is still in flight.
template <typename T, bool kTwoShot, bool kResidual, bool kBulk>
__device__ __forceinline__ void multi_body(const Params& p, const void* const* resid) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [N][Q]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t G = (uint32_t)kClusterMaxRanks;
    const uint32_t j = cluster_ctarank();
    const uint32_t hosted = (N - j + G - 1) / G;  // ranks j, j + G, ...
    const uint32_t S = p.per_cta;
    const uint32_t Q = kTwoShot ? S / G : S;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint32_t mine = kTwoShot ? (npos > j * Q ? min(Q, npos - j * Q) : 0u) : npos;

    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, (kBulk ? N : N - hosted) * mine * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    if (kBulk) {
        cluster_wait();  // every peer's barrier exists before any copy completes on it
        const uint32_t t = threadIdx.x;
        if (kTwoShot) {
            const uint32_t m = t / G;
            const uint32_t q = t - m * G;
            const uint32_t len = npos > q * Q ? min(Q, npos - q * Q) : 0u;
            if (m < hosted && len != 0) {
                const uint32_t rank = j + m * G;
                if (q == j || drop != (int32_t)rank)
                    bulk_g2s_multicast(smem_u32(stage + rank * Q),
                                       (const char*)p.send[rank] + (uint64_t)(base + q * Q) * kVecBytes,
                                       len * (uint32_t)kVecBytes, my_bar, (uint16_t)(1u << q));
            }
        } else if (t < hosted) {
            const uint32_t rank = j + t * G;
            const uint16_t all = (uint16_t)((1u << G) - 1u);
            bulk_g2s_multicast(smem_u32(stage + rank * Q), (const char*)p.send[rank] + (uint64_t)base * kVecBytes,
                               npos * (uint32_t)kVecBytes, my_bar,
                               drop != (int32_t)rank ? all : (uint16_t)(1u << j));
        }
    }
    // item it = (hosted rank m, vector v)
    const uint32_t items = hosted * npos;
    uint4 x[kClusterBatch];
    auto load_batch = [&](uint32_t b0) {
#pragma unroll
        for (int k = 0; k < kClusterBatch; ++k) {
            const uint32_t it = b0 + threadIdx.x + (uint32_t)k * nt;
            if (it >= items) continue;
            const uint32_t m = it / npos;
            x[k] = load_input<T>(p.send[j + m * G], base + (it - m * npos), p.count);
        }
    };
    if (!kBulk) {
        load_batch(0);
        cluster_wait();  // every peer's barrier exists before anyone stores into it
    }

    const uint32_t step = nt * (uint32_t)kClusterBatch;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < (kBulk ? 0u : items); b0 += step) {
        if (b0 != 0) load_batch(b0);
#pragma unroll
        for (int k = 0; k < kClusterBatch; ++k) {
            const uint32_t it = b0 + threadIdx.x + (uint32_t)k * nt;
            if (it >= items) continue;
            const uint32_t m = it / npos;
            const uint32_t v = it - m * npos;
            const uint32_t rank = j + m * G;
            const bool pushes = drop != (int32_t)rank;
            if (kTwoShot) {
                const uint32_t q = v / Q;
                const uint32_t u = v - q * Q;
                if (q == j) stage[rank * Q + u] = x[k];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(stage + rank * Q + u), q), x[k], map_to_rank(my_bar, q));
            } else {
                if (pushes) {
#pragma unroll 1
                    for (uint32_t c = 1; c < G; ++c) {
                        const uint32_t q = j + c < G ? j + c : j + c - G;
                        st_async_v4(map_to_rank(smem_u32(stage + rank * Q + v), q), x[k], map_to_rank(my_bar, q));
                    }
                }
                stage[rank * Q + v] = x[k];
            }
        }
    }
    if (!kBulk) cluster_arrive_relaxed();  // "my pushes are issued" (orders no data)
    int ok = 1;
    {
        Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, (int)j, 0);
        while (!mbar_try_wait(my_bar, 0u)) {
            if (waiter_expired(w)) {
                ok = 0;
                break;
            }
        }
    }
    if (kBulk) cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    __syncthreads();  // the hosted ranks' slots were written by other threads
    if (ok) {
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * Q + u]);
            // output of rank d at vector pos: the sum, or the sum plus d's residual
            auto emit = [&](uint32_t d, uint32_t pos) {
                if (kResidual) {
                    typename M::Acc a = acc;
                    M::add(a, load_input<T>(resid[d], pos, p.count));
                    store_output<T>(p.recv[d], pos, p.count, M::store(a));
                } else {
                    store_output<T>(p.recv[d], pos, p.count, M::store(acc));
                }
            };
            if (kTwoShot) {
#pragma unroll 1
                for (uint32_t d = 0; d < N; ++d) emit(d, base + j * Q + u);
            } else {
#pragma unroll 1
                for (uint32_t m = 0; m < hosted; ++m) emit(j + m * G, base + u);
            }
        }
    }
    if (kBulk) cluster_wait();  // every CTA's incoming bytes are in: none of my copies is still in flight
    else if (!__all_sync(0xffffffffu, ok)) cluster_wait();  // a thread whose wait ran out keeps the memory alive
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

template <typename T, bool kTwoShot, bool kBulk>
__global__ void __launch_bounds__(256) cluster_multi_kernel(const __grid_constant__ Params p) {
    multi_body<T, kTwoShot, false, kBulk>(p, nullptr);
}

template <typename T, bool kTwoShot>
__global__ void __launch_bounds__(256) residual_multi_kernel(const __grid_constant__ FusedParams f) {
    multi_body<T, kTwoShot, true, false>(f.base, f.resid);
}

// Persistent, double-buffered two-shot (the pages' double buffering, Sec. IV,
// in which receiving from a peer is what permits the next send to it,
// restated with mbarriers).  Cluster c handles
// slices c, c + G, c + 2G, ... (G clusters in the grid, p.nsteps slices in
// all); slice k of a cluster uses stage buffer b = k & 1.  Per buffer, each
// CTA has a "full" mbarrier (completed by the N-1 incoming partitions'
// bytes) and an "empty" mbarrier (N-1 arrivals: one from every receiver of
// this CTA's pushes, made once that receiver has consumed the buffer).  A
// sender pushes slice k >= 2 into buffer b only after its own empty[b] has
// seen every receiver finish slice k - 2.  Each thread loads the next
// slice's inputs before it waits on the current one, so HBM reads overlap
// the exchange, the reduction and the stores.
template <typename T>
__global__ void __launch_bounds__(256) cluster_pipe_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [2][N][Q] payload vectors
    __shared__ __align__(8) uint64_t full[2];
    __shared__ __align__(8) uint64_t empty[2];
    pdl_release_early();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t Q = S / N;
    const uint32_t G = (uint32_t)p.ctas_per_rank;  // clusters in the grid
    const uint32_t nslices = p.nsteps;
    const uint32_t nt = blockDim.x;
    const void* src = p.send[r];

    uint32_t s = cluster_id();
    uint4 x[kClusterBatch];
    {
        const uint32_t base = s * S;
        const uint32_t npos = min(S, p.nvec - base);
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = threadIdx.x + (uint32_t)j * nt;
            x[j] = make_uint4(0, 0, 0, 0);
            if (v < npos) x[j] = load_input<T>(src, base + v, p.count);
        }
    }
    const int32_t drop = p.drop_rank;
    const uint32_t full0 = smem_u32(&full[0]);    // full[b] at full0 + 8 b
    const uint32_t empty0 = smem_u32(&empty[0]);  // empty[b] at empty0 + 8 b
    if (threadIdx.x == 0) {
        mbar_init(full0, 1u);
        mbar_init(full0 + 8u, 1u);
        mbar_init(empty0, N - 1);
        mbar_init(empty0 + 8u, N - 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster_sync();  // every peer's barriers exist before anyone uses them

    Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, (int)r, 0);
#pragma unroll 1
    for (uint32_t k = 0; s < nslices; s += G, ++k) {
        const uint32_t b = k & 1u;
        const uint32_t base = s * S;
        const uint32_t npos = min(S, p.nvec - base);
        const uint32_t mine = npos > r * Q ? min(Q, npos - r * Q) : 0u;
        uint4* const buf = stage + b * N * Q;
        const uint32_t full_b = full0 + 8u * b;
        const uint32_t empty_b = empty0 + 8u * b;
        w.step = (int)k;
        if (threadIdx.x == 0) mbar_expect_tx(full_b, (N - 1) * mine * (uint32_t)kVecBytes);
        // credit: every receiver has consumed this buffer's previous slice
        if (k >= 2) {
            const bool ok = mbar_wait_bounded(empty_b, ((k - 2) >> 1) & 1u, w);
            if (!__syncthreads_and(ok)) break;
        }
        // push: partition q of my slice into slot [r] of CTA q's buffer b
        const uint32_t slot_r = smem_u32(buf + r * Q);
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = threadIdx.x + (uint32_t)j * nt;
            if (v >= npos) continue;
            const uint32_t q = v / Q;
            const uint32_t u = v - q * Q;
            if (q == r) {
                buf[r * Q + u] = x[j];
            } else if (drop != (int32_t)r) {
                st_async_v4(map_to_rank(slot_r + u * (uint32_t)kVecBytes, q), x[j], map_to_rank(full_b, q));
            }
        }
        // next slice's inputs, in flight during the wait, reduction and stores
        const uint32_t s_next = s + G;
        if (s_next < nslices) {
            const uint32_t nbase = s_next * S;
            const uint32_t nnpos = min(S, p.nvec - nbase);
#pragma unroll
            for (int j = 0; j < kClusterBatch; ++j) {
                const uint32_t v = threadIdx.x + (uint32_t)j * nt;
                if (v < nnpos) x[j] = load_input<T>(src, nbase + v, p.count);
            }
        }
        {
            const bool ok = mbar_wait_bounded(full_b, (k >> 1) & 1u, w);
            if (!__syncthreads_and(ok)) break;  // also makes my own slot visible
        }
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(buf[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, buf[q * Q + u]);
            const uint4 out = M::store(acc);
            const uint32_t pos = base + r * Q + u;
#pragma unroll 1
            for (uint32_t d0 = 0; d0 < N; ++d0) {
                const uint32_t d = r + d0 < N ? r + d0 : r + d0 - N;
                store_output<T>(p.recv[d], pos, p.count, out);
            }
        }
        __syncthreads();  // every read of buffer b is done
        if (threadIdx.x == 0 && s + 2 * G < nslices) {
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) {
                const uint32_t peer = r + q < N ? r + q : r + q - N;
                mbar_arrive_remote(map_to_rank(empty_b, peer));
            }
        }
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still store into its shared memory
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

template <typename T, bool kTrace>
static const void* cluster_kernel_for(int mode) {
    switch (mode) {
        case kClusterOneshot: return (const void*)cluster_kernel<T, false, kTrace>;
        case kClusterTwoshot: return (const void*)cluster_kernel<T, true, kTrace>;
        case kClusterTwoshotPipe: return (const void*)cluster_pipe_kernel<T>;
        case kClusterOneshotMulti: return (const void*)cluster_multi_kernel<T, false, false>;
        case kClusterTwoshotMulti: return (const void*)cluster_multi_kernel<T, true, false>;
        case kClusterOneshotMultiTma: return (const void*)cluster_multi_kernel<T, false, true>;
        case kClusterTwoshotMultiTma: return (const void*)cluster_multi_kernel<T, true, true>;
        case kClusterOneshotMultiRes: return (const void*)residual_multi_kernel<T, false>;
        case kClusterTwoshotMultiRes: return (const void*)residual_multi_kernel<T, true>;
        case kClusterOneshotTma: return (const void*)cluster_tma_kernel<T, false, kTrace>;
        case kClusterTwoshotTma: return (const void*)cluster_tma_kernel<T, true, kTrace>;
        case kClusterOneshotTmaRes: return (const void*)cluster_tma_residual_kernel<T, kTrace>;
    }
    return nullptr;
}

// trace: the variant with trace points (a trace buffer is set); the
// persistent and many-rank kernels have none.
static const void* cluster_kernel_ptr(rra_dtype_t dtype, int mode, bool trace = false) {
    switch (dtype) {
        case RRA_FP32: return trace ? cluster_kernel_for<float, true>(mode) : cluster_kernel_for<float, false>(mode);
        case RRA_BF16:
            return trace ? cluster_kernel_for<__nv_bfloat16, true>(mode) : cluster_kernel_for<__nv_bfloat16, false>(mode);
        case RRA_FP64: return trace ? cluster_kernel_for<double, true>(mode) : cluster_kernel_for<double, false>(mode);
    }
    return nullptr;
}

// Opt the kernel in to the full stage and to clusters of up to 16 CTAs.
static cudaError_t configure(const void* k) { return configure_cluster_kernel(k, (int)kClusterStageBytes); }

size_t cluster_stage_bytes(const Params& p, int mode) {
    const size_t n = (size_t)p.nranks;
    switch (mode) {
        case kClusterOneshot:
        case kClusterOneshotTma:
        case kClusterOneshotTmaRes: return n * p.per_cta * kVecBytes;
        case kClusterTwoshot:
        case kClusterTwoshotTma: return (size_t)p.per_cta / n * n * kVecBytes;
        case kClusterTwoshotPipe: return 2 * ((size_t)p.per_cta / n * n) * kVecBytes;
        case kClusterOneshotMulti:
        case kClusterOneshotMultiTma:
        case kClusterOneshotMultiRes: return n * p.per_cta * kVecBytes;
        case kClusterTwoshotMulti:
        case kClusterTwoshotMultiTma:
        case kClusterTwoshotMultiRes: return n * ((size_t)p.per_cta / kClusterMaxRanks) * kVecBytes;
    }
    return 0;
}

static bool is_multi(int mode) {
    return mode == kClusterOneshotMulti || mode == kClusterTwoshotMulti || mode == kClusterOneshotMultiRes ||
           mode == kClusterTwoshotMultiRes || mode == kClusterOneshotMultiTma || mode == kClusterTwoshotMultiTma;
}

// CTAs per cluster: one per rank, or 16 hosting several ranks each.
static unsigned cluster_ctas(int mode, int nranks) {
    return is_multi(mode) ? (unsigned)kClusterMaxRanks : (unsigned)nranks;
}

// `arg` is the kernel's parameter block: `p` itself, or the FusedParams
// that starts with it (residual modes).
static cudaError_t launch_cluster_args(const Params& p, void* arg, rra_dtype_t dtype, int mode, int threads,
                                       cudaStream_t stream, bool pdl) {
    const size_t smem = cluster_stage_bytes(p, mode);
    const bool multi = is_multi(mode);
    if (smem == 0 || smem > kClusterStageBytes || p.nranks < 2 || p.nranks > (multi ? kMaxRanks : kClusterMaxRanks))
        return cudaErrorInvalidValue;
    if (multi && p.nranks <= kClusterMaxRanks) return cudaErrorInvalidValue;
    if ((mode == kClusterTwoshot || mode == kClusterTwoshotPipe || mode == kClusterTwoshotTma) &&
        p.per_cta % (uint32_t)p.nranks != 0)
        return cudaErrorInvalidValue;
    if ((mode == kClusterTwoshotTma || mode == kClusterOneshotTma || mode == kClusterOneshotTmaRes) &&
        threads < p.nranks)
        return cudaErrorInvalidValue;  // the two-shot's copies are issued by threads 0..N-1
    if ((mode == kClusterTwoshotMulti || mode == kClusterTwoshotMultiRes || mode == kClusterTwoshotMultiTma) &&
        p.per_cta % (uint32_t)kClusterMaxRanks != 0)
        return cudaErrorInvalidValue;
    {   // the many-rank bulk copies are issued by threads 0 .. hosted x (16 or 1) - 1
        const int hosted = (p.nranks + kClusterMaxRanks - 1) / kClusterMaxRanks;
        if ((mode == kClusterTwoshotMultiTma && threads < hosted * kClusterMaxRanks) ||
            (mode == kClusterOneshotMultiTma && threads < hosted))
            return cudaErrorInvalidValue;
    }
    if (mode == kClusterTwoshotPipe && p.per_cta > (uint32_t)threads * kClusterBatch) return cudaErrorInvalidValue;
    const void* k = cluster_kernel_ptr(dtype, mode, p.trace != nullptr);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = configure(k);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    const unsigned cdim = cluster_ctas(mode, p.nranks);
    cfg.gridDim = dim3(cdim * (unsigned)p.ctas_per_rank);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cdim;
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
    void* args[] = {arg};
    return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch_cluster(const Params& p, rra_dtype_t dtype, int mode, int threads, cudaStream_t stream, bool pdl) {
    if (mode == kClusterOneshotMultiRes || mode == kClusterTwoshotMultiRes || mode == kClusterOneshotTmaRes)
        return cudaErrorInvalidValue;
    return launch_cluster_args(p, (void*)&p, dtype, mode, threads, stream, pdl);
}

cudaError_t launch_cluster_residual(const FusedParams& f, rra_dtype_t dtype, bool two_shot, int threads,
                                    cudaStream_t stream, bool pdl) {
    const int mode = two_shot ? kClusterTwoshotMultiRes : kClusterOneshotMultiRes;
    return launch_cluster_args(f.base, (void*)&f, dtype, mode, threads, stream, pdl);
}

cudaError_t launch_cluster_tma_residual(const FusedParams& f, rra_dtype_t dtype, int threads, cudaStream_t stream,
                                        bool pdl) {
    return launch_cluster_args(f.base, (void*)&f, dtype, kClusterOneshotTmaRes, threads, stream, pdl);
}

// Clusters of `nranks` CTAs of this kernel, `threads` threads and `smem`
// bytes of stage each, that can be resident at once (0 = this cluster shape
// cannot run on the device).
int cluster_max_active(rra_dtype_t dtype, int mode, int nranks, int threads, size_t smem) {
    const void* k = cluster_kernel_ptr(dtype, mode);
    if (k == nullptr || configure(k) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    const unsigned cdim = cluster_ctas(mode, nranks);
    cfg.gridDim = dim3(cdim);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cdim;
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
