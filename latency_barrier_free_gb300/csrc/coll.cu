// coll.cu -- ReduceScatter, AllGather, Broadcast and Reduce through
// distributed shared memory.
//
// "Every Microsecond Matters", Sec. III-A (opening): AllReduce is commonly
// built from ReduceScatter + AllGather or Reduce + Broadcast; the paper's
// review (summary) notes that the same barrier-free primitives serve these
// collectives.  Here they use the primitives of the cluster AllReduce
// (cluster.cu): one thread-block cluster of N CTAs per slice, CTA r = rank r,
// a push is an st.async into a peer's shared memory that completes the
// peer's mbarrier, and the only wait is a bounded wait on one's own mbarrier
// (data arrival is the signal, Sec. IV).  A CTA reads only its own rank's
// input and writes only its own rank's output -- except the bulk-copy
// Reduce, whose partition owners push their sums into the root's output.
//
// Layout (v = 16-byte vector, S = slice of p.per_cta vectors, nv = p.nvec
// vectors per block of `count` elements):
//   ReduceScatter  send[r] = N blocks of count; CTA r pushes block q's slice
//                  to CTA q's slot [r]; CTA q adds the N slots in rank order
//                  into recv[q].
//   AllGather      CTA r pushes its slice to slot [r] of every peer; CTA r
//                  writes slot p into block p of recv[r], for every p.
//   Broadcast      the root CTA pushes its slice to slot [0] of every peer
//                  and writes its own output from registers.
//   Reduce         every CTA but the root's pushes its slice to the root's
//                  slot [r]; the root adds in rank order into recv[root].
//                  With bulk copies: CTA r copies partition q of its slice
//                  to CTA q's slot [r]; CTA q adds in rank order into
//                  partition q of recv[root].
// Blocks start at element q * count, which is not 16-byte aligned when count
// is not a multiple of the elements per vector; such vectors are moved
// element by element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cluster_prims.cuh"
#include "prims.cuh"
#include "rra_internal.h"
#include "kernel_attrs.h"

namespace rra {
namespace {

template <typename T>
struct Bits;
template <>
struct Bits<__nv_bfloat16> { using U = uint16_t; };
template <>
struct Bits<float> { using U = uint32_t; };
template <>
struct Bits<double> { using U = uint64_t; };

// Vector u of a block of `count` elements that starts at element `elem0` of
// `base`; elements past the block's end read as zero.
template <typename T>
__device__ __forceinline__ uint4 load_block(const void* base, uint64_t elem0, uint32_t u, uint64_t count) {
    constexpr int VE = VecMath<T>::kElems;
    using U = typename Bits<T>::U;
    const uint64_t e = (uint64_t)u * VE;
    const uint64_t first = elem0 + e;
    if (e + VE <= count && first % VE == 0) return ld_input_v4((const T*)base + first);
    union {
        uint4 v;
        U x[VE];
    } w;
    w.v = make_uint4(0u, 0u, 0u, 0u);
    const int n = (int)min((uint64_t)VE, count - e);
    const U* s = (const U*)base + first;
    for (int i = 0; i < n; ++i) w.x[i] = s[i];
    return w.v;
}

// Store vector u of such a block; only elements inside the block are written.
template <typename T>
__device__ __forceinline__ void store_block(void* base, uint64_t elem0, uint32_t u, uint64_t count, uint4 v) {
    constexpr int VE = VecMath<T>::kElems;
    using U = typename Bits<T>::U;
    const uint64_t e = (uint64_t)u * VE;
    const uint64_t first = elem0 + e;
    if (e + VE <= count && first % VE == 0) {
        st_output_v4((T*)base + first, v);
        return;
    }
    union {
        uint4 v;
        U x[VE];
    } w;
    w.v = v;
    const int n = (int)min((uint64_t)VE, count - e);
    U* d = (U*)base + first;
    for (int i = 0; i < n; ++i) d[i] = w.x[i];
}

}  // namespace

template <typename T, int kOp>
__global__ void __launch_bounds__(256) coll_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [slots][S]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint32_t root = (uint32_t)p.root;
    const uint64_t count = p.count;
    const bool is_root = r == root;

    // bytes this CTA receives, and input vectors it reads
    uint32_t incoming = 0, items = 0;
    switch (kOp) {
        case kCollReduceScatter: incoming = (N - 1) * npos; items = N * npos; break;
        case kCollAllGather: incoming = (N - 1) * npos; items = npos; break;
        case kCollBroadcast: incoming = is_root ? 0u : npos; items = is_root ? npos : 0u; break;
        case kCollReduce: incoming = is_root ? (N - 1) * npos : 0u; items = npos; break;
    }
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, incoming * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const void* src = p.send[r];
    const int32_t drop = p.drop_rank;
    const bool pushes = drop != (int32_t)r;

    // input item v: block q = v / npos (ReduceScatter; else 0), vector u
    uint4 x[kClusterBatch];
    auto load_batch = [&](uint32_t b0) {
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v >= items) continue;
            const uint32_t q = kOp == kCollReduceScatter ? v / npos : 0u;
            const uint32_t u = v - q * npos;
            x[j] = load_block<T>(src, (uint64_t)q * count, base + u, count);
        }
    };
    load_batch(0);
    cluster_wait();  // every peer's barrier exists before anyone stores into it

    const uint32_t step = nt * (uint32_t)kClusterBatch;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < items; b0 += step) {
        if (b0 != 0) load_batch(b0);
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v >= items) continue;
            if (kOp == kCollReduceScatter) {
                const uint32_t q = v / npos;
                const uint32_t u = v - q * npos;
                if (q == r) stage[r * S + u] = x[j];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(stage + r * S + u), q), x[j], map_to_rank(my_bar, q));
            } else if (kOp == kCollAllGather) {
                stage[r * S + v] = x[j];
                if (pushes) {
#pragma unroll 1
                    for (uint32_t k = 1; k < N; ++k) {
                        const uint32_t q = r + k < N ? r + k : r + k - N;
                        st_async_v4(map_to_rank(smem_u32(stage + r * S + v), q), x[j], map_to_rank(my_bar, q));
                    }
                }
            } else if (kOp == kCollBroadcast) {  // root only
                if (pushes) {
#pragma unroll 1
                    for (uint32_t k = 1; k < N; ++k) {
                        const uint32_t q = r + k < N ? r + k : r + k - N;
                        st_async_v4(map_to_rank(smem_u32(stage + v), q), x[j], map_to_rank(my_bar, q));
                    }
                }
                store_block<T>(p.recv[r], 0, base + v, count, x[j]);
            } else {  // Reduce
                if (is_root) stage[r * S + v] = x[j];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(stage + r * S + v), root), x[j], map_to_rank(my_bar, root));
            }
        }
    }
    cluster_arrive_relaxed();  // "my pushes are issued" (orders no data)

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
    __syncthreads();  // own slot written by other threads of this CTA
    if (ok) {
        if (kOp == kCollReduceScatter || (kOp == kCollReduce && is_root)) {
#pragma unroll 1
            for (uint32_t u = threadIdx.x; u < npos; u += nt) {
                typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
                for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * S + u]);
                store_block<T>(p.recv[r], 0, base + u, count, M::store(acc));
            }
        } else if (kOp == kCollAllGather) {
#pragma unroll 1
            for (uint32_t v = threadIdx.x; v < N * npos; v += nt) {
                const uint32_t q = v / npos;
                const uint32_t u = v - q * npos;
                store_block<T>(p.recv[r], (uint64_t)q * count, base + u, count, stage[q * S + u]);
            }
        } else if (kOp == kCollBroadcast && !is_root) {
#pragma unroll 1
            for (uint32_t u = threadIdx.x; u < npos; u += nt) store_block<T>(p.recv[r], 0, base + u, count, stage[u]);
        }
    }
    cluster_wait();  // every peer has issued its pushes into this CTA's shared memory
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// AllGather and Broadcast up to 16 ranks with the push made by the TMA
// engine: one multicast bulk copy per slice from the sender's input into
// slot [r] of every CTA's window (AllGather) or into slot [0] (Broadcast,
// from the root; the root's own window included), completing each CTA's
// mbarrier.  Every CTA then writes its output from its window.  Whole
// 16-byte vectors are copied: the last vector of an input whose size is not
// a multiple of 16 bytes is read in full (it lies in the same 16-byte block,
// so the same page, as valid data) and its extra lanes are never stored.  A
// CTA leaves after a cluster barrier that every CTA reaches once its own
// bytes are in, so no copy it issued is still in flight.
// kStoreBulk: the window goes to the output by bulk copies too (one per
// block, issued by thread 0, waited for before the CTA leaves) instead of
// vector stores by every thread; the host chooses it only when every output
// is device memory of this GPU and a block is a whole number of 16-byte
// vectors (so no copy writes past its block).
template <typename T, int kOp, bool kStoreBulk>
__global__ void __launch_bounds__(256) coll_bulk_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) uint4 stage[];  // AllGather [N][S], Broadcast [S]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint32_t root = (uint32_t)p.root;
    const uint64_t count = p.count;
    const uint32_t incoming = kOp == kCollAllGather ? N * npos : npos;  // vectors, the own copy included
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, incoming * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    cluster_wait();  // every peer's barrier exists before any copy completes on it
    if (threadIdx.x == 0 && (kOp == kCollAllGather || r == root)) {
        const uint16_t mask = drop != (int32_t)r ? (uint16_t)((1u << N) - 1u) : (uint16_t)(1u << r);
        bulk_g2s_multicast(smem_u32(stage + (kOp == kCollAllGather ? r * S : 0u)),
                           (const char*)p.send[r] + (size_t)base * kVecBytes, npos * (uint32_t)kVecBytes, my_bar,
                           mask);
    }
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
    cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    if (ok && kStoreBulk) {
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            constexpr uint32_t nblk = kOp == kCollAllGather ? kClusterMaxRanks : 1u;
            const uint64_t block_bytes = count * sizeof(T);
#pragma unroll 1
            for (uint32_t q = 0; q < nblk && q < N; ++q)
                bulk_s2g((char*)p.recv[r] + q * block_bytes + (uint64_t)base * kVecBytes,
                         smem_u32(stage + (kOp == kCollAllGather ? q * S : 0u)), npos * (uint32_t)kVecBytes);
            bulk_s2g_commit_wait();
        }
    } else if (ok) {
        if (kOp == kCollAllGather) {
#pragma unroll 1
            for (uint32_t v = threadIdx.x; v < N * npos; v += nt) {
                const uint32_t q = v / npos;
                const uint32_t u = v - q * npos;
                store_block<T>(p.recv[r], (uint64_t)q * count, base + u, count, stage[q * S + u]);
            }
        } else {
#pragma unroll 1
            for (uint32_t u = threadIdx.x; u < npos; u += nt) store_block<T>(p.recv[r], 0, base + u, count, stage[u]);
        }
    }
    cluster_wait();  // every CTA's bytes are in: none of my copies is still in flight
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// ReduceScatter up to 16 ranks with the push made by the TMA engine: thread
// q of CTA r copies the slice of block q of rank r's input into slot [r] of
// CTA q's window (one bulk copy, completing CTA q's mbarrier; q = r is the
// own slot).  CTA q then adds its N slots in rank order into recv[q].  The
// host chooses it only when every input is device memory of this GPU and a
// block is a whole number of 16-byte vectors, so that every copy starts on a
// 16-byte boundary and reads its block alone.  The CTA leaves after a
// cluster barrier that every CTA reaches once its own bytes are in.
template <typename T>
__global__ void __launch_bounds__(256) coll_rs_bulk_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [N][S]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint64_t count = p.count;
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, N * npos * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    cluster_wait();  // every peer's barrier exists before any copy completes on it
    {
        const uint32_t q = threadIdx.x;
        if (q < N && (q == r || drop != (int32_t)r))
            bulk_g2s_multicast(smem_u32(stage + r * S),
                               (const char*)p.send[r] + q * count * sizeof(T) + (uint64_t)base * kVecBytes,
                               npos * (uint32_t)kVecBytes, my_bar, (uint16_t)(1u << q));
    }
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
    cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    if (ok) {
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < npos; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * S + u]);
            store_block<T>(p.recv[r], 0, base + u, count, M::store(acc));
        }
    }
    cluster_wait();  // every CTA's bytes are in: none of my copies is still in flight
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// Reduce up to 16 ranks with the push made by the TMA engine, in the
// ReduceScatter pattern of the two-shot: a slice of S = N * Q vectors is
// split into N partitions of Q, and thread q of CTA r copies partition q of
// rank r's slice into slot [r] of CTA q's window (one bulk copy completing
// CTA q's mbarrier; q = r is the own slot).  CTA q adds its N slots in rank
// order and stores the sums straight into partition q of the root's output
// (a push of the reduced partition to the root), so no CTA carries more than
// its partition and there is no second exchange.  The input is one block at
// send[r], so every copy starts on a 16-byte boundary; the host chooses this
// kernel only when every input is device memory of this GPU.
template <typename T>
__global__ void __launch_bounds__(256) coll_reduce_bulk_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [N][Q]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t Q = S / N;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint64_t count = p.count;
    // vectors of partition q of this slice
    auto part_len = [&](uint32_t q) -> uint32_t { return npos > q * Q ? min(Q, npos - q * Q) : 0u; };
    const uint32_t mine = part_len(r);
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, N * mine * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    cluster_wait();  // every peer's barrier exists before any copy completes on it
    {
        const uint32_t q = threadIdx.x;
        const uint32_t len = q < N ? part_len(q) : 0u;
        if (len != 0 && (q == r || drop != (int32_t)r))
            bulk_g2s_multicast(smem_u32(stage + r * Q),
                               (const char*)p.send[r] + (uint64_t)(base + q * Q) * kVecBytes,
                               len * (uint32_t)kVecBytes, my_bar, (uint16_t)(1u << q));
    }
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
    cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    if (ok) {
        void* const out = p.recv[p.root];
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * Q + u]);
            store_block<T>(out, 0, base + r * Q + u, count, M::store(acc));
        }
    }
    cluster_wait();  // every CTA's bytes are in: none of my copies is still in flight
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// Reduce above 16 ranks with the push made by the TMA engine, in the
// partition pattern of coll_reduce_bulk_kernel on 16-CTA clusters: a slice of
// S = 16 Q vectors is split into 16 partitions, and thread (m, q) of CTA j
// copies partition q of hosted rank m's slice into slot [rank] of CTA q's
// window; CTA q adds its N slots in rank order and stores the sums into
// partition q of the root's output.  No CTA carries more than its partition.
template <typename T>
__global__ void __launch_bounds__(256) coll_reduce_multi_bulk_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];  // [N][Q]
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t G = (uint32_t)kClusterMaxRanks;
    const uint32_t j = cluster_ctarank();
    const uint32_t hosted = (N - j + G - 1) / G;  // ranks j, j + G, ...
    const uint32_t S = p.per_cta;
    const uint32_t Q = S / G;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint64_t count = p.count;
    auto part_len = [&](uint32_t q) -> uint32_t { return npos > q * Q ? min(Q, npos - q * Q) : 0u; };
    const uint32_t mine = part_len(j);
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, N * mine * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    cluster_wait();  // every peer's barrier exists before any copy completes on it
#pragma unroll 1
    for (uint32_t c = threadIdx.x; c < hosted * G; c += nt) {
        const uint32_t m = c / G;
        const uint32_t q = c - m * G;
        const uint32_t rank = j + m * G;
        const uint32_t len = part_len(q);
        if (len != 0 && (q == j || drop != (int32_t)rank))
            bulk_g2s_multicast(smem_u32(stage + rank * Q),
                               (const char*)p.send[rank] + (uint64_t)(base + q * Q) * kVecBytes,
                               len * (uint32_t)kVecBytes, my_bar, (uint16_t)(1u << q));
    }
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
    cluster_arrive_relaxed();  // "my incoming bytes are in" (or my wait ran out)
    if (ok) {
        void* const out = p.recv[p.root];
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
            for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * Q + u]);
            store_block<T>(out, 0, base + j * Q + u, count, M::store(acc));
        }
    }
    cluster_wait();  // every CTA's bytes are in: none of my copies is still in flight
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// The same four collectives for nranks > 16 (clusters hold at most 16
// CTAs): a cluster of G = 16 CTAs per slice, CTA j acting for ranks j,
// j + G, j + 2G, ... (as the many-rank cluster AllReduce).  A push to a rank
// hosted by the same CTA is a plain shared-memory store; to another CTA, an
// st.async that completes that CTA's mbarrier, which expects the bytes of
// every rank it does not host.  Slots are indexed by rank as above; a
// ReduceScatter CTA keeps one set of N slots per hosted owner.
// kBulk: every push is a TMA bulk copy from the input (device memory of this
// GPU, checked by the host), the own CTA's slots included: ReduceScatter one
// copy per hosted rank and owner (blocks of whole 16-byte vectors only),
// AllGather one multicast copy per hosted rank, Broadcast one from the root's
// CTA.  Each CTA then writes from its window, the root's CTA of a Broadcast
// included.  (The bulk-copy Reduce is coll_reduce_multi_bulk_kernel.)
// kStoreBulk (AllGather, Broadcast, with kBulk): the window goes to the
// hosted ranks' outputs by bulk copies (one per hosted rank and block,
// spread over the threads, each waited for by its issuing thread); the host
// chooses it only when every output is device memory of this GPU and a
// block is whole 16-byte vectors.
template <typename T, int kOp, bool kBulk, bool kStoreBulk>
__global__ void __launch_bounds__(256) coll_multi_kernel(const __grid_constant__ Params p) {
    static_assert(!(kBulk && kOp == kCollReduce), "the bulk-copy Reduce is coll_reduce_multi_bulk_kernel");
    static_assert(!kStoreBulk || (kBulk && (kOp == kCollAllGather || kOp == kCollBroadcast)),
                  "bulk stores: AllGather and Broadcast on bulk copies");
    using M = VecMath<T>;
    extern __shared__ __align__(16) uint4 stage[];
    __shared__ __align__(8) uint64_t bar;
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t G = (uint32_t)kClusterMaxRanks;
    const uint32_t j = cluster_ctarank();
    const uint32_t hosted = (N - j + G - 1) / G;  // ranks j, j + G, ...
    const uint32_t S = p.per_cta;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint32_t root = (uint32_t)p.root;
    const uint32_t root_cta = root % G;
    const uint64_t count = p.count;
    const bool root_here = j == root_cta;

    // bytes this CTA receives, and input items (hosted rank, block, vector) it reads
    uint32_t incoming = 0, items = 0;
    switch (kOp) {
        case kCollReduceScatter: incoming = hosted * (N - hosted) * npos; items = hosted * N * npos; break;
        case kCollAllGather: incoming = (N - hosted) * npos; items = hosted * npos; break;
        case kCollBroadcast: incoming = root_here ? 0u : npos; items = root_here ? npos : 0u; break;
        case kCollReduce: incoming = root_here ? (N - hosted) * npos : 0u; items = hosted * npos; break;
    }
    if (kBulk) {  // every slot arrives by copy, the own CTA's included
        switch (kOp) {
            case kCollReduceScatter: incoming = hosted * N * npos; break;
            case kCollAllGather: incoming = N * npos; break;
            case kCollBroadcast: incoming = npos; break;
        }
    }
    const uint32_t my_bar = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(my_bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(my_bar, incoming * (uint32_t)kVecBytes);
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const int32_t drop = p.drop_rank;
    const uint32_t per_rank = kOp == kCollReduceScatter ? N * npos : npos;  // items per hosted rank

    uint4 x[kClusterBatch];
    auto load_batch = [&](uint32_t b0) {
#pragma unroll
        for (int k = 0; k < kClusterBatch; ++k) {
            const uint32_t it = b0 + threadIdx.x + (uint32_t)k * nt;
            if (it >= items) continue;
            if (kOp == kCollBroadcast) {
                x[k] = load_block<T>(p.send[root], 0, base + it, count);
            } else {
                const uint32_t m = it / per_rank;
                const uint32_t rem = it - m * per_rank;
                const uint32_t q = kOp == kCollReduceScatter ? rem / npos : 0u;
                x[k] = load_block<T>(p.send[j + m * G], (uint64_t)q * count, base + (rem - q * npos), count);
            }
        }
    };
    if (kBulk) {
        cluster_wait();  // every peer's barrier exists before any copy completes on it
        const uint16_t all = (uint16_t)((1u << G) - 1u);
        const uint32_t vbytes = npos * (uint32_t)kVecBytes;
        const uint32_t ncopies = kOp == kCollReduceScatter ? hosted * N
                                 : kOp == kCollBroadcast   ? (root_here ? 1u : 0u)
                                                           : hosted;  // AllGather
#pragma unroll 1
        for (uint32_t c = threadIdx.x; c < ncopies; c += nt) {
            if (kOp == kCollReduceScatter) {  // block q's slice of hosted rank m to owner q's CTA
                const uint32_t m = c / N;
                const uint32_t q = c - m * N;
                const uint32_t rank = j + m * G;
                const uint32_t dst = q % G;
                if (dst == j || drop != (int32_t)rank)
                    bulk_g2s_multicast(smem_u32(stage + ((q / G) * N + rank) * S),
                                       (const char*)p.send[rank] + q * count * sizeof(T) + (uint64_t)base * kVecBytes,
                                       vbytes, my_bar, (uint16_t)(1u << dst));
            } else if (kOp == kCollAllGather) {  // hosted rank c's slice into its slot of every CTA
                const uint32_t rank = j + c * G;
                bulk_g2s_multicast(smem_u32(stage + rank * S), (const char*)p.send[rank] + (uint64_t)base * kVecBytes,
                                   vbytes, my_bar, drop != (int32_t)rank ? all : (uint16_t)(1u << j));
            } else if (kOp == kCollBroadcast) {  // the root's slice into slot [0] of every CTA
                bulk_g2s_multicast(smem_u32(stage), (const char*)p.send[root] + (uint64_t)base * kVecBytes, vbytes,
                                   my_bar, drop != (int32_t)root ? all : (uint16_t)(1u << j));
            }
        }
    } else {
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
            if (kOp == kCollBroadcast) {  // root's CTA: every other CTA's slot [0], and the hosted outputs
                if (drop != (int32_t)root) {
#pragma unroll 1
                    for (uint32_t c = 1; c < G; ++c) {
                        const uint32_t q = j + c < G ? j + c : j + c - G;
                        st_async_v4(map_to_rank(smem_u32(stage + it), q), x[k], map_to_rank(my_bar, q));
                    }
                }
#pragma unroll 1
                for (uint32_t m = 0; m < hosted; ++m) store_block<T>(p.recv[j + m * G], 0, base + it, count, x[k]);
                continue;
            }
            const uint32_t m = it / per_rank;
            const uint32_t rem = it - m * per_rank;
            const uint32_t rank = j + m * G;
            const bool pushes = drop != (int32_t)rank;
            if (kOp == kCollReduceScatter) {
                const uint32_t q = rem / npos;  // owner rank of this block
                const uint32_t u = rem - q * npos;
                const uint32_t c = q % G;
                uint4* const slot = stage + ((q / G) * N + rank) * S + u;
                if (c == j) *slot = x[k];
                else if (pushes) st_async_v4(map_to_rank(smem_u32(slot), c), x[k], map_to_rank(my_bar, c));
            } else if (kOp == kCollAllGather) {
                stage[rank * S + rem] = x[k];
                if (pushes) {
#pragma unroll 1
                    for (uint32_t c = 1; c < G; ++c) {
                        const uint32_t q = j + c < G ? j + c : j + c - G;
                        st_async_v4(map_to_rank(smem_u32(stage + rank * S + rem), q), x[k], map_to_rank(my_bar, q));
                    }
                }
            } else {  // Reduce
                if (root_here) stage[rank * S + rem] = x[k];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(stage + rank * S + rem), root_cta), x[k],
                                map_to_rank(my_bar, root_cta));
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
    __syncthreads();  // slots of hosted ranks written by other threads of this CTA
    if (ok) {
        if (kOp == kCollReduceScatter) {
#pragma unroll 1
            for (uint32_t it = threadIdx.x; it < hosted * npos; it += nt) {
                const uint32_t m = it / npos;
                const uint32_t u = it - m * npos;
                const uint4* const slots = stage + m * N * S + u;
                typename M::Acc acc = M::load(slots[0]);
#pragma unroll 1
                for (uint32_t q = 1; q < N; ++q) M::add(acc, slots[q * S]);
                store_block<T>(p.recv[j + m * G], 0, base + u, count, M::store(acc));
            }
        } else if (kOp == kCollReduce) {
            if (root_here) {
#pragma unroll 1
                for (uint32_t u = threadIdx.x; u < npos; u += nt) {
                    typename M::Acc acc = M::load(stage[u]);
#pragma unroll 1
                    for (uint32_t q = 1; q < N; ++q) M::add(acc, stage[q * S + u]);
                    store_block<T>(p.recv[root], 0, base + u, count, M::store(acc));
                }
            }
        } else if (kStoreBulk) {  // AllGather / Broadcast: one bulk copy per hosted rank (and block)
            fence_proxy_async_smem();
            const uint32_t blocks = kOp == kCollAllGather ? N : 1u;
            const uint64_t block_bytes = count * sizeof(T);
#pragma unroll 1
            for (uint32_t c = threadIdx.x; c < hosted * blocks; c += nt) {
                const uint32_t m = c / blocks;
                const uint32_t q = c - m * blocks;
                bulk_s2g((char*)p.recv[j + m * G] + q * block_bytes + (uint64_t)base * kVecBytes,
                         smem_u32(stage + q * S), npos * (uint32_t)kVecBytes);
            }
            bulk_s2g_commit_wait();
        } else if (kOp == kCollAllGather) {
#pragma unroll 1
            for (uint32_t it = threadIdx.x; it < hosted * N * npos; it += nt) {
                const uint32_t m = it / (N * npos);
                const uint32_t v = it - m * N * npos;
                const uint32_t q = v / npos;
                const uint32_t u = v - q * npos;
                store_block<T>(p.recv[j + m * G], (uint64_t)q * count, base + u, count, stage[q * S + u]);
            }
        } else if (kBulk || !root_here) {  // Broadcast (the root's CTA wrote its outputs unless kBulk)
#pragma unroll 1
            for (uint32_t it = threadIdx.x; it < hosted * npos; it += nt) {
                const uint32_t m = it / npos;
                const uint32_t u = it - m * npos;
                store_block<T>(p.recv[j + m * G], 0, base + u, count, stage[u]);
            }
        }
    }
    cluster_wait();  // every peer has issued its pushes into this CTA's shared memory
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

// Broadcast and Reduce in two hops, for large slices: the root's CTA would
// otherwise send (Broadcast) or receive (Reduce) (N-1) S vectors alone.  The
// slice is cut into N parts of Q = S / N vectors (part q = CTA q's).
//   Broadcast: the root pushes part q to CTA q (region A); every CTA then
//     pushes its part to every CTA but the root (region B slot [r]); each
//     writes its output from its part and region B.  The root writes its
//     output from its input.
//   Reduce: ReduceScatter (rank r pushes part q to CTA q's region A slot
//     [r]); CTA q adds part q in rank order and pushes it to the root's
//     region B slot [q]; the root writes its output.  Same rank-order sums.
// Region A, then region B, in shared memory; one mbarrier per region.
template <typename T, int kOp>
__global__ void __launch_bounds__(256) coll_split_kernel(const __grid_constant__ Params p) {
    using M = VecMath<T>;
    constexpr bool kBcast = kOp == kCollBroadcastSplit;
    extern __shared__ __align__(16) uint4 stage[];
    __shared__ __align__(8) uint64_t bars[2];
    pdl_release_early();
    const uint32_t N = (uint32_t)p.nranks;
    const uint32_t r = cluster_ctarank();
    const uint32_t S = p.per_cta;
    const uint32_t Q = S / N;
    const uint32_t base = cluster_id() * S;
    const uint32_t npos = min(S, p.nvec - base);
    const uint32_t nt = blockDim.x;
    const uint32_t root = (uint32_t)p.root;
    const uint64_t count = p.count;
    const bool is_root = r == root;
    auto len_of = [&](uint32_t q) { return npos > q * Q ? min(Q, npos - q * Q) : 0u; };
    const uint32_t mine = len_of(r);
    uint4* const regA = stage;
    uint4* const regB = stage + (kBcast ? Q : N * Q);
    const uint32_t barA = smem_u32(&bars[0]);
    const uint32_t barB = smem_u32(&bars[1]);
    if (threadIdx.x == 0) {
        mbar_init(barA, 1u);
        mbar_init(barB, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (kBcast) {
            mbar_expect_tx(barA, (is_root ? 0u : mine) * (uint32_t)kVecBytes);
            mbar_expect_tx(barB, (is_root ? 0u : npos - mine) * (uint32_t)kVecBytes);
        } else {
            mbar_expect_tx(barA, (N - 1) * mine * (uint32_t)kVecBytes);
            mbar_expect_tx(barB, (is_root ? npos - mine : 0u) * (uint32_t)kVecBytes);
        }
    }
    cluster_arrive_relaxed();
    pdl_wait();
    const uint64_t t_start = globaltimer_ns();
    const void* src = p.send[r];
    const bool pushes = p.drop_rank != (int32_t)r;
    const uint32_t items = kBcast ? (is_root ? npos : 0u) : npos;
    uint4 x[kClusterBatch];
    auto load_batch = [&](uint32_t b0) {
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v < items) x[j] = load_input<T>(src, base + v, count);
        }
    };
    load_batch(0);
    cluster_wait();  // every peer's barriers exist

    // hop 1: part q of the slice to CTA q
    const uint32_t step = nt * (uint32_t)kClusterBatch;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < items; b0 += step) {
        if (b0 != 0) load_batch(b0);
#pragma unroll
        for (int j = 0; j < kClusterBatch; ++j) {
            const uint32_t v = b0 + threadIdx.x + (uint32_t)j * nt;
            if (v >= items) continue;
            const uint32_t q = v / Q;
            const uint32_t u = v - q * Q;
            if (kBcast) {
                store_output<T>(p.recv[r], base + v, count, x[j]);  // the root's own output
                if (q == r) regB[r * Q + u] = x[j];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(regA + u), q), x[j], map_to_rank(barA, q));
            } else {
                if (q == r) regA[r * Q + u] = x[j];
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(regA + r * Q + u), q), x[j], map_to_rank(barA, q));
            }
        }
    }
    int ok = 1;
    Waiter w = make_waiter(t_start, p.timeout_ns, p.ctrl, (int)r, 0);
    while (!mbar_try_wait(barA, 0u))
        if (waiter_expired(w)) {
            ok = 0;
            break;
        }
    ok = __syncthreads_and(ok);  // also: this CTA's own part, written by other threads
    // hop 2
    if (ok) {
#pragma unroll 1
        for (uint32_t u = threadIdx.x; u < mine; u += nt) {
            if (kBcast) {
                const uint4 y = is_root ? regB[r * Q + u] : regA[u];
                if (!is_root) store_output<T>(p.recv[r], base + r * Q + u, count, y);
                if (pushes) {
#pragma unroll 1
                    for (uint32_t k = 1; k < N; ++k) {
                        const uint32_t q = r + k < N ? r + k : r + k - N;
                        if (q != root)
                            st_async_v4(map_to_rank(smem_u32(regB + r * Q + u), q), y, map_to_rank(barB, q));
                    }
                }
            } else {
                typename M::Acc acc = M::load(regA[u]);
#pragma unroll 1
                for (uint32_t q = 1; q < N; ++q) M::add(acc, regA[q * Q + u]);
                const uint4 out = M::store(acc);
                if (is_root) store_output<T>(p.recv[r], base + r * Q + u, count, out);
                else if (pushes)
                    st_async_v4(map_to_rank(smem_u32(regB + r * Q + u), root), out, map_to_rank(barB, root));
            }
        }
    }
    cluster_arrive_relaxed();  // "my pushes are issued"
    if (ok) {
        w.step = 1;
        while (!mbar_try_wait(barB, 0u))
            if (waiter_expired(w)) {
                ok = 0;
                break;
            }
    }
    ok = __syncthreads_and(ok);
    // the other parts into this CTA's output (Broadcast: every CTA but the
    // root's; Reduce: the root's)
    if (ok && (kBcast ? !is_root : is_root)) {
#pragma unroll 1
        for (uint32_t v = threadIdx.x; v < npos; v += nt) {
            const uint32_t q = v / Q;
            if (q == r) continue;
            store_output<T>(p.recv[r], base + v, count, regB[v]);
        }
    }
    if (!ok) cluster_wait();  // a CTA whose wait ran out keeps its memory until every peer has pushed
    if (p.timing != nullptr && threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        p.timing[2 * blockIdx.x] = t_start;
        p.timing[2 * blockIdx.x + 1] = t_end;
    }
}

template <typename T, bool kBulk>
static const void* coll_multi_for(int op, bool store_bulk) {
    switch (op) {
        case kCollReduceScatter: return (const void*)coll_multi_kernel<T, kCollReduceScatter, kBulk, false>;
        case kCollAllGather:
            if (kBulk && store_bulk) return (const void*)coll_multi_kernel<T, kCollAllGather, true, true>;
            return (const void*)coll_multi_kernel<T, kCollAllGather, kBulk, false>;
        case kCollBroadcast:
            if (kBulk && store_bulk) return (const void*)coll_multi_kernel<T, kCollBroadcast, true, true>;
            return (const void*)coll_multi_kernel<T, kCollBroadcast, kBulk, false>;
        case kCollReduce:
            return kBulk ? (const void*)coll_reduce_multi_bulk_kernel<T>
                         : (const void*)coll_multi_kernel<T, kCollReduce, false, false>;
    }
    return nullptr;
}

template <typename T>
static const void* coll_kernel_for(int op, bool multi, bool bulk = false, bool store_bulk = false) {
    if (multi) return bulk ? coll_multi_for<T, true>(op, store_bulk) : coll_multi_for<T, false>(op, false);
    switch (op) {
        case kCollReduceScatter: return (const void*)coll_kernel<T, kCollReduceScatter>;
        case kCollAllGather: return (const void*)coll_kernel<T, kCollAllGather>;
        case kCollBroadcast: return (const void*)coll_kernel<T, kCollBroadcast>;
        case kCollReduce: return (const void*)coll_kernel<T, kCollReduce>;
        case kCollBroadcastSplit: return (const void*)coll_split_kernel<T, kCollBroadcastSplit>;
        case kCollReduceSplit: return (const void*)coll_split_kernel<T, kCollReduceSplit>;
    }
    return nullptr;
}

// ReduceScatter, AllGather, Broadcast and Reduce have bulk-copy kernels at
// every rank count (ReduceScatter only for blocks of whole 16-byte vectors);
// the bulk stores of AllGather and Broadcast exist up to 16 ranks.
bool coll_has_bulk(int op, int nranks) {
    return (op == kCollReduceScatter || op == kCollAllGather || op == kCollBroadcast || op == kCollReduce) &&
           nranks >= 2 && nranks <= kMaxRanks;
}

const char* coll_kernel_name(int op, int nranks, bool bulk, bool store_bulk) {
    static const char* const kBulk[] = {"coll_bulk_kernel<reduce_scatter>", "coll_bulk_kernel<all_gather>",
                                        "coll_bulk_kernel<broadcast>", "coll_bulk_kernel<reduce>"};
    static const char* const kBulkStore[] = {"", "coll_bulk_kernel<all_gather, bulk store>",
                                             "coll_bulk_kernel<broadcast, bulk store>", ""};
    static const char* const kPlain[] = {"coll_kernel<reduce_scatter>", "coll_kernel<all_gather>",
                                         "coll_kernel<broadcast>", "coll_kernel<reduce>"};
    static const char* const kMulti[] = {"coll_multi_kernel<reduce_scatter>", "coll_multi_kernel<all_gather>",
                                         "coll_multi_kernel<broadcast>", "coll_multi_kernel<reduce>"};
    if (op < 0 || op > kCollReduceSplit) return "unknown";
    if (op == kCollBroadcastSplit) return "coll_split_kernel<broadcast>";
    if (op == kCollReduceSplit) return "coll_split_kernel<reduce>";
    static const char* const kMultiBulk[] = {"coll_multi_kernel<reduce_scatter, bulk>", "coll_multi_kernel<all_gather, bulk>",
                                             "coll_multi_kernel<broadcast, bulk>", "coll_reduce_multi_bulk_kernel"};
    static const char* const kMultiBulkStore[] = {"", "coll_multi_kernel<all_gather, bulk, bulk store>",
                                                  "coll_multi_kernel<broadcast, bulk, bulk store>", ""};
    if (bulk && coll_has_bulk(op, nranks) && nranks > kClusterMaxRanks)
        return store_bulk ? kMultiBulkStore[op] : kMultiBulk[op];
    if (bulk && coll_has_bulk(op, nranks)) return store_bulk ? kBulkStore[op] : kBulk[op];
    return nranks > kClusterMaxRanks ? kMulti[op] : kPlain[op];
}

template <typename T>
static const void* coll_bulk_for(int op, bool store_bulk) {
    if (op == kCollReduceScatter) return (const void*)coll_rs_bulk_kernel<T>;
    if (op == kCollReduce) return (const void*)coll_reduce_bulk_kernel<T>;
    if (store_bulk)
        return op == kCollAllGather ? (const void*)coll_bulk_kernel<T, kCollAllGather, true>
                                    : (const void*)coll_bulk_kernel<T, kCollBroadcast, true>;
    return op == kCollAllGather ? (const void*)coll_bulk_kernel<T, kCollAllGather, false>
                                : (const void*)coll_bulk_kernel<T, kCollBroadcast, false>;
}

static const void* coll_kernel_ptr(rra_dtype_t dtype, int op, int nranks, bool bulk, bool store_bulk = false) {
    const bool multi = nranks > kClusterMaxRanks;
    if (bulk && multi && coll_has_bulk(op, nranks)) {
        switch (dtype) {
            case RRA_FP32: return coll_kernel_for<float>(op, true, true, store_bulk);
            case RRA_BF16: return coll_kernel_for<__nv_bfloat16>(op, true, true, store_bulk);
            case RRA_FP64: return coll_kernel_for<double>(op, true, true, store_bulk);
        }
        return nullptr;
    }
    if (bulk && coll_has_bulk(op, nranks)) {
        switch (dtype) {
            case RRA_FP32: return coll_bulk_for<float>(op, store_bulk);
            case RRA_BF16: return coll_bulk_for<__nv_bfloat16>(op, store_bulk);
            case RRA_FP64: return coll_bulk_for<double>(op, store_bulk);
        }
        return nullptr;
    }
    switch (dtype) {
        case RRA_FP32: return coll_kernel_for<float>(op, multi);
        case RRA_BF16: return coll_kernel_for<__nv_bfloat16>(op, multi);
        case RRA_FP64: return coll_kernel_for<double>(op, multi);
    }
    return nullptr;
}

// CTAs per cluster: one per rank up to 16 ranks, 16 above.
static int coll_cdim(int nranks) { return nranks < kClusterMaxRanks ? nranks : kClusterMaxRanks; }

// Opt the kernel in to the full stage and to clusters of up to 16 CTAs.
static cudaError_t configure_coll(const void* k) { return configure_cluster_kernel(k, (int)kClusterStageBytes); }

size_t coll_stage_bytes(const Params& p, int op) {
    const size_t n = (size_t)p.nranks;
    const size_t q = p.per_cta / n;  // split forms: vectors per part
    if (p.nranks > kClusterMaxRanks) {  // hosted ranks: CTA 0 hosts the most
        const size_t hosted = (n + kClusterMaxRanks - 1) / kClusterMaxRanks;
        switch (op) {
            case kCollReduceScatter: return hosted * n * p.per_cta * kVecBytes;
            case kCollBroadcast: return (size_t)p.per_cta * kVecBytes;
            case kCollAllGather:
            case kCollReduce: return n * p.per_cta * kVecBytes;
            default: return 0;  // no split forms
        }
    }
    switch (op) {
        case kCollBroadcast: return (size_t)p.per_cta * kVecBytes;
        case kCollBroadcastSplit: return (q + n * q) * kVecBytes;
        case kCollReduceSplit: return 2 * n * q * kVecBytes;
        default: return n * p.per_cta * kVecBytes;
    }
}

cudaError_t launch_coll(const Params& p, rra_dtype_t dtype, int op, int threads, cudaStream_t stream, bool pdl,
                        bool bulk, bool store_bulk) {
    // the bulk-copy Reduce holds N partitions of S / N vectors: S vectors
    const bool part_reduce = bulk && op == kCollReduce && p.nranks <= kClusterMaxRanks;  // coll_reduce_bulk_kernel
    const bool multi_reduce = bulk && op == kCollReduce && p.nranks > kClusterMaxRanks;  // coll_reduce_multi_bulk_kernel
    const size_t smem = part_reduce    ? (size_t)p.per_cta * kVecBytes
                        : multi_reduce ? (size_t)p.nranks * (p.per_cta / kClusterMaxRanks) * kVecBytes
                                       : coll_stage_bytes(p, op);
    if (smem == 0 || smem > kClusterStageBytes || p.nranks < 2 || p.nranks > kMaxRanks || p.root < 0 ||
        p.root >= p.nranks)
        return cudaErrorInvalidValue;
    if ((op == kCollBroadcastSplit || op == kCollReduceSplit || part_reduce) &&
        p.per_cta % (uint32_t)p.nranks != 0)
        return cudaErrorInvalidValue;
    if (multi_reduce && p.per_cta % (uint32_t)kClusterMaxRanks != 0) return cudaErrorInvalidValue;
    const int cdim = coll_cdim(p.nranks);
    const uint64_t es = dtype == RRA_BF16 ? 2u : dtype == RRA_FP64 ? 8u : 4u;
    if (store_bulk && (!bulk || !coll_has_bulk(op, p.nranks) || op == kCollReduceScatter || op == kCollReduce ||
                       (p.count * es) % kVecBytes != 0))
        return cudaErrorInvalidValue;  // a bulk copy would write past its block
    if (bulk && op == kCollReduceScatter && (p.count * es) % kVecBytes != 0)
        return cudaErrorInvalidValue;  // a block would start off a 16-byte boundary
    const void* k = coll_kernel_ptr(dtype, op, p.nranks, bulk, store_bulk);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = configure_coll(k);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cdim * p.ctas_per_rank));  // ctas_per_rank: clusters (slices)
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cdim;
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

int coll_max_active(rra_dtype_t dtype, int op, int nranks, int threads, size_t smem, bool bulk) {
    const void* k = coll_kernel_ptr(dtype, op, nranks, bulk);
    if (k == nullptr || configure_coll(k) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int cdim = coll_cdim(nranks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cdim);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)cdim;
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
