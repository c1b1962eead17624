// kernels.cu -- the four barrier-free AllReduce kernels and the window
// initialiser.
//
// Source: "Every Microsecond Matters: Achieving Near Speed-of-Light Latency in
// GPU Collectives" (arXiv 2607.16100): Sec. III-A (one-shot push and two-shot
// AllReduce), Sec. IV (LL, sentinel, bidirectional double buffering, Fig. 4)
// and Fig. 5 (two-shot LL128 atomic AllReduce).
//
// Execution model.  One cooperative launch of N * C CTAs; CTA b is sub-slice
// c = b % C of virtual rank r = b / C.  Rank r reads only send[r] and its own
// window, and writes only peers' windows and recv[r].  All scratch traffic is
// 16-byte vectors.  No CTA ever waits at a grid-wide barrier: every wait is a
// poll on data (LL flag, sentinel, or LL128 line counter), bounded in time.
//
// Credit (double buffering, Sec. IV).  Step k of a call uses scratch parity
// (epoch + k) & 1, so a slot is reused two steps later.  The position -> thread
// map is the same in every step of a call, so the thread that fills slot
// position v of peer p at step k+2 is the thread that, at step k+1, received
// p's data for position v -- which p's corresponding thread sent only after it
// had consumed (and, for sentinels, reset) position v of step k.  A
// fence.acq_rel.gpu at the start of every step (when a call has >= 3 steps)
// turns that chain into release/acquire pairs.  Between calls, the kernel
// boundary orders everything.
//
// Summation order.  One-shot and two-shot add the N contributions of an
// element in rank order 0..N-1 (binary32 running value for binary32 and
// bfloat16, binary64 for binary64): the result is deterministic and equals the
// fixed-order definition bit for bit.  LL128-atomic adds with L2 atomics in
// arrival order (the paper notes the non-determinism).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "prims.cuh"
#include "rra_internal.h"

namespace rra {

// ------------------------------------------------------------ helpers ----
__device__ __forceinline__ char* window(const Params& p, int r) {
    return p.win0 + (uint64_t)r * p.stride;
}

// Per-CTA prologue/epilogue shared by all kernels.
struct CtaState {
    uint64_t epoch;  // epoch of step 0 of this call (0 when the call needs none)
    uint64_t t_start;
    int rank, sub;
    bool skip;       // earlier device error, or epoch wrap: do nothing
    bool drop;       // injected fault: do not store to peers
    bool advance;    // the call uses epochs: advance them at exit
};

// Epoch scrub (once per kScrubPeriod steps).  Every CTA of the co-resident
// grid zeroes its share of all LL flag regions, then the grid meets at one
// bounded barrier: the only grid-wide wait in the library, taken once every
// 2^31 steps and never on the per-call path.
__device__ __noinline__ bool epoch_scrub(const Params& p, int rank) {
    __shared__ int s_ok;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t n1 = p.ll_bytes / 16, n2 = p.llag_bytes / 16;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int nwin = p.scrub_ranks > 0 ? p.scrub_ranks : p.nranks;
    for (int q = 0; q < nwin; ++q) {
        char* wq = p.win0 + (uint64_t)q * p.stride;
        for (uint64_t i = tid; i < n1; i += nthreads) st_relaxed_v4(wq + p.ll_off + i * 16, z);
        for (uint64_t i = tid; i < n2; i += nthreads) st_relaxed_v4(wq + p.llag_off + i * 16, z);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t gen = ld_relaxed_u32(&p.ctrl->scrub_gen);
        fence_acq_rel_gpu();  // release this CTA's zeroes; the gen read before the arrival
        const uint32_t arrived = atomicAdd(&p.ctrl->scrub_arrive, 1u) + 1u;
        if (arrived == gridDim.x) {
            st_relaxed_u32(&p.ctrl->scrub_arrive, 0u);
            fence_acq_rel_gpu();
            st_relaxed_u32(&p.ctrl->scrub_gen, gen + 1u);
        } else {
            Waiter w = make_waiter(globaltimer_ns(), p.timeout_ns, p.ctrl, rank, -2);
            while (ld_relaxed_u32(&p.ctrl->scrub_gen) == gen) {
                if (waiter_expired(w)) { ok = 0; break; }
            }
        }
        fence_acq_rel_gpu();  // acquire every CTA's zeroes
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Every thread reads the control words itself (one broadcast line per warp),
// so the first input loads overlap this round trip instead of waiting behind
// a block barrier.  The barrier sits in the epilogue instead: no thread may
// overwrite epoch slot b before every thread of the CTA has read it.
// Programmatic dependent launch (prims.cuh): release the next kernel on the
// stream (at entry for a one-cluster grid, else after the wait), and wait
// until the previous kernel has completed and its memory is visible before
// this one touches global memory.  Both are no-ops without the launch
// attribute.  Kernels without their own prologue call this first.
__device__ __forceinline__ void pdl_entry() {
    pdl_release_early();
    pdl_wait();
}

// The parameter fields the AllReduce kernels use, read once before the kernel
// waits for its predecessor (griddepcontrol.wait): a first read of a
// parameter line misses the constant cache (about 0.1 us each on GB300), and
// these misses are then paid while the previous kernel drains instead of one
// after another on the critical path.  Touches no global memory.
__device__ __forceinline__ void warm_params(const Params& p) {
    const unsigned r = blockIdx.x / (unsigned)p.ctas_per_rank;
    asm volatile("" : : "l"(p.win0), "l"(p.ctrl), "l"(p.timing), "l"(p.trace), "l"(p.stride), "l"(p.count),
                 "l"(p.timeout_ns), "l"(p.region_off), "l"(p.slot_bytes), "l"(p.parity_bytes), "l"(p.aux_off));
    asm volatile("" : : "r"(p.nvec), "r"(p.chunk_vecs), "r"(p.per_cta), "r"(p.nsteps), "r"(p.nranks),
                 "r"(p.epoch_slots), "r"(p.drop_rank), "l"(p.send[r]), "l"(p.recv[r]));
}

// need_epoch: the call uses epochs (LL flags, or the parity of a multi-step
// call's double buffering).  A single-step call on sentinel slots needs none:
// at a call boundary every sentinel slot is idle, so it uses parity 0, reads
// no epoch and leaves the epoch unchanged.
__device__ __forceinline__ CtaState cta_prologue(const Params& p, bool need_epoch = true) {
    CtaState s;
    s.t_start = globaltimer_ns();
    s.rank = (int)(blockIdx.x / (unsigned)p.ctas_per_rank);
    s.sub = (int)(blockIdx.x % (unsigned)p.ctas_per_rank);
    s.advance = need_epoch;
    s.epoch = need_epoch ? ld_relaxed_u64(&p.ctrl->epoch_m1[blockIdx.x]) + 1ull : 0ull;
    const uint32_t status = ld_relaxed_u32(&p.ctrl->status);
    s.skip = status != 0u;
    s.drop = p.drop_rank == s.rank;
    // The epochs of this call are [epoch, epoch + nsteps); if they would reach
    // the next multiple of kScrubPeriod, scrub first and restart one past it.
    // The test depends only on the epoch, which every thread of every CTA
    // reads equal, so the whole grid takes this branch together.
    if (need_epoch && (s.epoch & (kScrubPeriod - 1)) + (uint64_t)p.nsteps + 1ull >= kScrubPeriod) {
        if (epoch_scrub(p, s.rank)) s.epoch = (s.epoch | (kScrubPeriod - 1)) + 2ull;
        else s.skip = true;
    }
    return s;
}

__device__ __forceinline__ void cta_epilogue(const Params& p, const CtaState& s) {
    __syncthreads();  // every thread has read its epoch slot
    if (!s.skip && s.advance) {
        // Advance every epoch slot this CTA owns: slots b, b + G, b + 2G, ...
        // Plain stores: the slots are read only by later kernels, after the
        // kernel boundary (or griddepcontrol.wait) has made them visible.
        const uint64_t next_m1 = s.epoch + p.nsteps - 1ull;
        const unsigned G = gridDim.x;
        for (unsigned slot = blockIdx.x + threadIdx.x * G; slot < (unsigned)p.epoch_slots;
             slot += blockDim.x * G) {
            st_weak_u64(&p.ctrl->epoch_m1[slot], next_m1);
        }
    }
    if (threadIdx.x == 0) {
        const uint64_t t_end = globaltimer_ns();
        if (p.timing != nullptr) {  // both stamps at the end: no store on the timed path
            p.timing[2 * blockIdx.x] = s.t_start;
            p.timing[2 * blockIdx.x + 1] = t_end;
        }
        if (p.trace != nullptr) {
            p.trace[(uint64_t)blockIdx.x * kTracePoints] = s.t_start;
            p.trace[(uint64_t)blockIdx.x * kTracePoints + 5] = t_end;
        }
    }
}

constexpr int kBatch = 4;  // sources polled with loads in flight at once

// Poll one scratch vector once.  LL: both LL lines carry `ep` in all four
// flags.  Sentinel: no atomic unit still holds the sentinel.
template <typename T, bool kLL>
__device__ __forceinline__ bool poll_once(const char* slot_pos, uint32_t ep, uint4& out) {
    if (kLL) return ll_load(slot_pos, ep, out);
    out = ld_scratch<VecMath<T>::kUnitBytes>(slot_pos);
    return sentinel_arrived<VecMath<T>::kUnitBytes>(out);
}

// Polling the slots of sources q0 .. q0+kBatch-1 of one position (skipping
// `skip`, sources at or beyond n, and sources whose `limit` is not above the
// position): `poll_issue` sends all loads at once, `poll_finish` spins on the
// ones not yet arrived.  Callers issue the batches of two positions before
// finishing either, so their round trips overlap.  poll_finish returns false
// if the wait gave up.
struct NoLimit {
    __device__ __forceinline__ bool operator()(int) const { return true; }
};

template <typename T, bool kLL, typename Has = NoLimit>
__device__ __forceinline__ void poll_issue(const char* slot0, uint64_t slot_stride, int q0, int n, int skip,
                                           uint32_t ep, uint4 (&val)[kBatch], bool (&ok)[kBatch],
                                           Has has = Has()) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        const int q = q0 + j;
        ok[j] = true;
        if (q < n && q != skip && has(q)) ok[j] = poll_once<T, kLL>(slot0 + (uint64_t)q * slot_stride, ep, val[j]);
    }
}

template <typename T, bool kLL>
__device__ __forceinline__ bool poll_finish(const char* slot0, uint64_t slot_stride, int q0, uint32_t ep,
                                            Waiter& w, uint4 (&val)[kBatch], bool (&ok)[kBatch]) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        const int q = q0 + j;
        while (!ok[j]) {
            if (waiter_expired(w)) return false;
            ok[j] = poll_once<T, kLL>(slot0 + (uint64_t)q * slot_stride, ep, val[j]);
        }
    }
    return true;
}

template <typename T, bool kLL>
__device__ __forceinline__ bool poll_batch(const char* slot0, uint64_t slot_stride, int q0, int n, int skip,
                                           uint32_t ep, Waiter& w, uint4 (&val)[kBatch]) {
    bool ok[kBatch];
    poll_issue<T, kLL>(slot0, slot_stride, q0, n, skip, ep, val, ok);
    return poll_finish<T, kLL>(slot0, slot_stride, q0, ep, w, val, ok);
}

// One-shot push of this thread's positions v0, v0 + T, ... < end: the input
// loads of kPushPos positions are issued together, then each vector is stored
// into slot [parity][r] of every peer (consecutive lanes store consecutive
// vectors of the same peer window, so the stores coalesce).
constexpr int kPushPos = 4;

template <typename T, bool kLL>
__device__ __forceinline__ void push_positions(const Params& p, int r, uint32_t base, uint32_t v0, uint32_t end,
                                               uint64_t par_off, uint32_t ep, const uint4* pre = nullptr) {
    constexpr int U = VecMath<T>::kUnitBytes;
    constexpr uint32_t kPosBytes = kLL ? 2 * kVecBytes : kVecBytes;
    const uint32_t T_ = blockDim.x;
    const int N = p.nranks;
#pragma unroll 1
    for (; v0 < end; v0 += kPushPos * T_) {
        uint4 x[kPushPos];
#pragma unroll
        for (int j = 0; j < kPushPos; ++j) {
            const uint32_t v = v0 + (uint32_t)j * T_;
            if (v < end) x[j] = (j == 0 && pre != nullptr) ? *pre : load_input<T>(p.send[r], base + v, p.count);
        }
        pre = nullptr;
#pragma unroll
        for (int j = 0; j < kPushPos; ++j) {
            const uint32_t v = v0 + (uint32_t)j * T_;
            if (v >= end) break;
            char* dst = p.win0 + p.region_off + par_off + (uint64_t)r * p.slot_bytes + (uint64_t)v * kPosBytes;
#pragma unroll 1
            for (int q = 0; q < N; ++q, dst += p.stride) {
                if (q == r) continue;
                if (kLL) ll_store(dst, x[j], ep);
                else st_scratch<U>(dst, x[j]);
            }
        }
    }
}

// ---------------------------------------------------- one-shot (push) ----
// Sec. III-A "One-shot" in push mode + Sec. IV "LL" / "Sentinel"; the
// bcast() of Fig. 9: each rank stores its chunk into every peer's slot, then
// polls its own window for the N-1 incoming slots and reduces.  kTrace: the
// variant with the in-kernel trace points (rra_comm_set_trace), launched
// only when a trace buffer is set; without them the kernel's code is smaller
// and its latency-bound path measured up to 0.4 us shorter at 128 B.
template <typename T, bool kLL, bool kTrace>
__device__ __forceinline__ bool oneshot_body(const Params& p, const CtaState& s, const uint4* pre) {
    using M = VecMath<T>;
    constexpr int U = M::kUnitBytes;
    constexpr uint32_t kPosBytes = kLL ? 2 * kVecBytes : kVecBytes;
    const int N = p.nranks, r = s.rank;
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;
    const uint32_t pos1 = pos0 + p.per_cta;
    char* const mine = window(p, r) + p.region_off;
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);
    uint64_t* const tr = (kTrace && p.trace != nullptr && threadIdx.x == 0)
                             ? p.trace + (uint64_t)blockIdx.x * kTracePoints
                             : nullptr;
    if (tr) tr[1] = globaltimer_after(s.epoch + (uint64_t)s.skip);  // epoch and status words arrived

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t ep = (uint32_t)e;
        const uint64_t par_off = (e & 1ull) * p.parity_bytes;
        const uint32_t base = k * p.chunk_vecs;
        const uint32_t end = min(pos1, min(p.chunk_vecs, p.nvec - base));
        w.step = (int)k;
        if (k > 0 && p.nsteps > 2) fence_acq_rel_gpu();

        // push: my chunk into slot [parity][r] of every peer
        if (!s.drop) push_positions<T, kLL>(p, r, base, pos0 + threadIdx.x, end, par_off, ep, k == 0 ? pre : nullptr);
        if (tr && k == 0) tr[2] = globaltimer_ns();
        // receive: poll the N-1 incoming slots of two positions at a time,
        // reduce each in rank order
#pragma unroll 1
        for (uint32_t v = pos0 + threadIdx.x; v < end; v += 2 * blockDim.x) {
            const uint32_t v2 = v + blockDim.x;
            const bool two = v2 < end;
            const uint4 own = load_input<T>(p.send[r], base + v, p.count);
            const uint4 own2 = two ? load_input<T>(p.send[r], base + v2, p.count) : make_uint4(0, 0, 0, 0);
            char* const slot0 = mine + par_off + (uint64_t)v * kPosBytes;
            char* const slot2 = mine + par_off + (uint64_t)v2 * kPosBytes;
            typename M::Acc acc, acc2;
#pragma unroll 1
            for (int q0 = 0; q0 < N; q0 += kBatch) {
                uint4 val[kBatch], val2[kBatch];
                bool ok[kBatch], ok2[kBatch];
                poll_issue<T, kLL>(slot0, p.slot_bytes, q0, N, r, ep, val, ok);
                poll_issue<T, kLL>(slot2, p.slot_bytes, q0, two ? N : 0, r, ep, val2, ok2);
                if (!poll_finish<T, kLL>(slot0, p.slot_bytes, q0, ep, w, val, ok)) return false;
                if (!poll_finish<T, kLL>(slot2, p.slot_bytes, q0, ep, w, val2, ok2)) return false;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    if (q >= N) break;
                    const uint4 x = (q == r) ? own : val[j];
                    const uint4 x2 = (q == r) ? own2 : val2[j];
                    if (q == 0) {
                        acc = M::load(x);
                        acc2 = M::load(x2);
                    } else {
                        M::add(acc, x);
                        M::add(acc2, x2);
                    }
                }
            }
            const uint4 out = M::store(acc);
            if (tr && k == 0 && v == pos0) tr[3] = globaltimer_after(out.x);
            store_output<T>(p.recv[r], base + v, p.count, out);
            if (two) store_output<T>(p.recv[r], base + v2, p.count, M::store(acc2));
            if (tr && k == 0 && v == pos0) tr[4] = globaltimer_ns();
            // sentinel: the consumed slots back to the sentinel (after the
            // output, which is what the caller waits for)
            if (!kLL) {
#pragma unroll 1
                for (int q = 0; q < N; ++q) {
                    if (q == r) continue;
                    st_scratch<U>(slot0 + (uint64_t)q * p.slot_bytes, sentinel_vec());
                    if (two) st_scratch<U>(slot2 + (uint64_t)q * p.slot_bytes, sentinel_vec());
                }
            }
        }
    }
    return true;
}

// Wide variant for many ranks: the threads of a CTA split the (source,
// position) items of both the push and the poll, so a position's N-1 sources
// are polled by different threads at once (one round trip instead of N/4).
// Polled vectors are staged raw in shared memory; one thread per position
// then adds the N values in rank order, so the result is the same bit pattern
// as the narrow variant.  Positions are processed in rounds of `R` so the
// stage fits.  A thread that gives up raises a shared flag; the whole CTA
// leaves at the next block barrier.
constexpr int kStageVecs = kWideStageVecs;  // 48 KiB of shared memory

template <typename T, bool kLL>
__device__ __forceinline__ bool oneshot_wide_body(const Params& p, const CtaState& s, uint4* stage, int* fail,
                                                  const uint4* pre) {
    using M = VecMath<T>;
    constexpr int U = M::kUnitBytes;
    constexpr uint32_t kPosBytes = kLL ? 2 * kVecBytes : kVecBytes;
    const int N = p.nranks, r = s.rank;
    const uint32_t T_ = blockDim.x;
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;
    const uint32_t pos1 = pos0 + p.per_cta;
    const uint32_t R = (uint32_t)(kStageVecs / N);
    char* const mine = window(p, r) + p.region_off;
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t ep = (uint32_t)e;
        const uint64_t par_off = (e & 1ull) * p.parity_bytes;
        const uint32_t base = k * p.chunk_vecs;
        const uint32_t end = min(pos1, min(p.chunk_vecs, p.nvec - base));
        w.step = (int)k;
        if (k > 0 && p.nsteps > 2) fence_acq_rel_gpu();

        // push: thread per position, as in the narrow variant
        if (!s.drop) push_positions<T, kLL>(p, r, base, pos0 + threadIdx.x, end, par_off, ep, k == 0 ? pre : nullptr);
#pragma unroll 1
        for (uint32_t r0 = pos0; r0 < end; r0 += R) {
            const uint32_t rn = min(R, end - r0);
            const uint32_t items = rn * (uint32_t)N;
            // poll: item i = (source q = i / rn, position r0 + i % rn), kBatch in flight
#pragma unroll 1
            for (uint32_t i0 = threadIdx.x; i0 < items; i0 += kBatch * T_) {
                uint4 val[kBatch];
                bool ok[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const uint32_t i = i0 + (uint32_t)j * T_;
                    ok[j] = true;
                    if (i < items) {
                        const int q = (int)(i / rn);
                        const uint32_t v = r0 + i % rn;
                        if (q == r) val[j] = load_input<T>(p.send[r], base + v, p.count);
                        else ok[j] = poll_once<T, kLL>(mine + par_off + (uint64_t)q * p.slot_bytes +
                                                           (uint64_t)v * kPosBytes, ep, val[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const uint32_t i = i0 + (uint32_t)j * T_;
                    if (i >= items) break;
                    const int q = (int)(i / rn);
                    const uint32_t v = r0 + i % rn;
                    const char* slot = mine + par_off + (uint64_t)q * p.slot_bytes + (uint64_t)v * kPosBytes;
                    while (!ok[j] && *(volatile int*)fail == 0) {
                        if (waiter_expired(w)) { *(volatile int*)fail = 1; break; }
                        ok[j] = poll_once<T, kLL>(slot, ep, val[j]);
                    }
                    if (!ok[j]) break;
                    stage[(uint32_t)q * R + (i % rn)] = val[j];
                    if (!kLL && q != r) st_scratch<U>((char*)slot, sentinel_vec());
                }
            }
            __syncthreads();
            if (*(volatile int*)fail) return false;
            // reduce: one thread per position, sources in rank order
#pragma unroll 1
            for (uint32_t vl = threadIdx.x; vl < rn; vl += T_) {
                typename M::Acc acc = M::load(stage[vl]);
#pragma unroll 1
                for (int q = 1; q < N; ++q) M::add(acc, stage[(uint32_t)q * R + vl]);
                store_output<T>(p.recv[r], base + r0 + vl, p.count, M::store(acc));
            }
            __syncthreads();
        }
    }
    return true;
}

// The thread's first input vector of step 0, loaded before the control words
// are read so that the two round trips overlap (only a read of the caller's
// input, in bounds; unused if the call turns out to be skipped).
template <typename T>
__device__ __forceinline__ bool prefetch_first(const Params& p, uint4& pre) {
    const uint32_t sub = blockIdx.x % (unsigned)p.ctas_per_rank;
    const int rank = (int)(blockIdx.x / (unsigned)p.ctas_per_rank);
    const uint32_t v = sub * p.per_cta + threadIdx.x;
    const uint32_t end = min((sub + 1u) * p.per_cta, min(p.chunk_vecs, p.nvec));
    if (v >= end) return false;
    pre = load_input<T>(p.send[rank], v, p.count);
    return true;
}

// Address hints for the lines a one-shot thread touches first -- its input
// vector, its output, its slot in every peer window and the slots it polls in
// its own window (both parities: the epoch is not known yet), and the
// control words -- issued before the kernel waits for its predecessor.  A
// prefetch reads no data into the SM, so it may precede griddepcontrol.wait;
// it fills L2 and the address translations while the previous kernel drains.
// Small N only (N <= 8).
template <bool kLL>
__device__ __forceinline__ void prefetch_paths(const Params& p) {
    constexpr uint32_t kPosBytes = kLL ? 2 * kVecBytes : kVecBytes;
    const uint32_t sub = blockIdx.x % (unsigned)p.ctas_per_rank;
    const int r = (int)(blockIdx.x / (unsigned)p.ctas_per_rank);
    const uint32_t v = sub * p.per_cta + threadIdx.x;
    if (threadIdx.x == 0) {
        prefetch_l2(&p.ctrl->status);
        prefetch_l2(&p.ctrl->epoch_m1[blockIdx.x]);
    }
    if (p.nranks > 8 || v >= min((sub + 1u) * p.per_cta, min(p.chunk_vecs, p.nvec))) return;
    const uint64_t pos = (uint64_t)v * kPosBytes;
    prefetch_l2((const char*)p.send[r] + (uint64_t)v * kVecBytes);
    prefetch_l2((const char*)p.recv[r] + (uint64_t)v * kVecBytes);
    for (int q = 0; q < p.nranks; ++q) {
        if (q == r) continue;
        const char* peer = window(p, q) + p.region_off + (uint64_t)r * p.slot_bytes + pos;
        const char* mine = window(p, r) + p.region_off + (uint64_t)q * p.slot_bytes + pos;
        prefetch_l2(peer);
        prefetch_l2(mine);
        if (kLL || p.nsteps > 1) {
            prefetch_l2(peer + p.parity_bytes);
            prefetch_l2(mine + p.parity_bytes);
        }
    }
}

template <typename T, bool kLL, bool kTrace>
__global__ void __launch_bounds__(256) oneshot_kernel(const __grid_constant__ Params p) {
    pdl_release_early();
    warm_params(p);
    prefetch_paths<kLL>(p);
    pdl_wait();
    uint4 pre;
    const bool has_pre = prefetch_first<T>(p, pre);
    const CtaState s = cta_prologue(p, kLL || p.nsteps > 1);
    if (!s.skip) (void)oneshot_body<T, kLL, kTrace>(p, s, has_pre ? &pre : nullptr);
    cta_epilogue(p, s);
}

template <typename T, bool kLL>
__global__ void __launch_bounds__(256) oneshot_wide_kernel(const __grid_constant__ Params p) {
    __shared__ uint4 stage[kStageVecs];
    __shared__ int fail;
    pdl_release_early();
    warm_params(p);
    pdl_wait();
    uint4 pre;
    const bool has_pre = prefetch_first<T>(p, pre);
    if (threadIdx.x == 0) fail = 0;
    CtaState s = cta_prologue(p, kLL || p.nsteps > 1);
    s.skip = __syncthreads_or(s.skip) != 0;  // block barriers follow: skip must be CTA-uniform
    if (!s.skip) (void)oneshot_wide_body<T, kLL>(p, s, stage, &fail, has_pre ? &pre : nullptr);
    cta_epilogue(p, s);
}

// ----------------------------------------- barrier baseline (not barrier-free) ----
// The design the paper replaces ("Every Microsecond Matters", Sec. III-B and
// Fig. 3): plain stores, then a memory barrier among the peers, then reads,
// then a second barrier before the buffers may be reused.  The barrier is the
// pattern the paper measures with ncclLsaBarrierSession: a flag is written to
// every peer, then each participant waits for every peer's flag.  Here the
// participants are the CTAs with one sub-index c of all N ranks; thread q of
// the CTA signals and waits for peer q.  Flags carry a tag that only grows
// within an epoch scrub period, and arrival is tested as tag-difference >= 0
// because a fast peer may already have posted the next tag.
__device__ __forceinline__ bool flag_barrier(const Params& p, const CtaState& s, uint32_t tag, Waiter& w,
                                             int* fail) {
    __syncthreads();  // the CTA's data stores happen before the flag stores
    const int N = p.nranks, r = s.rank, q = (int)threadIdx.x;
    if (q < N && q != r) {
        fence_acq_rel_gpu();  // release
        if (!s.drop)
            st_relaxed_u32(window(p, q) + p.aux_off + ((uint64_t)s.sub * kMaxRanks + (uint64_t)r) * 4, tag);
        const char* flag = window(p, r) + p.aux_off + ((uint64_t)s.sub * kMaxRanks + (uint64_t)q) * 4;
        while ((int32_t)(ld_relaxed_u32(flag) - tag) < 0) {
            if (*(volatile int*)fail) break;
            if (waiter_expired(w)) { *(volatile int*)fail = 1; break; }
        }
        fence_acq_rel_gpu();  // acquire
    }
    __syncthreads();  // every peer's data before the CTA's reads
    return *(volatile int*)fail == 0;
}

template <typename T>
__device__ __forceinline__ bool oneshot_barrier_body(const Params& p, const CtaState& s, int* fail) {
    using M = VecMath<T>;
    const int N = p.nranks, r = s.rank;
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;
    const uint32_t pos1 = pos0 + p.per_cta;
    char* const mine = window(p, r) + p.region_off;
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t tag = (uint32_t)(2ull * e);
        const uint32_t base = k * p.chunk_vecs;
        const uint32_t end = min(pos1, min(p.chunk_vecs, p.nvec - base));
        w.step = (int)k;
        if (!s.drop) {
#pragma unroll 1
            for (uint32_t v = pos0 + threadIdx.x; v < end; v += blockDim.x) {
                const uint4 x = load_input<T>(p.send[r], base + v, p.count);
                char* dst = p.win0 + p.region_off + (uint64_t)r * p.slot_bytes + (uint64_t)v * kVecBytes;
#pragma unroll 1
                for (int q = 0; q < N; ++q, dst += p.stride) {
                    if (q != r) st_relaxed_v4(dst, x);
                }
            }
        }
        if (!flag_barrier(p, s, tag, w, fail)) return false;  // data ready everywhere
#pragma unroll 1
        for (uint32_t v = pos0 + threadIdx.x; v < end; v += blockDim.x) {
            const uint4 own = load_input<T>(p.send[r], base + v, p.count);
            const char* const slot0 = mine + (uint64_t)v * kVecBytes;
            typename M::Acc acc;
#pragma unroll 1
            for (int q0 = 0; q0 < N; q0 += kBatch) {
                uint4 val[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    if (q < N && q != r) val[j] = ld_relaxed_v4(slot0 + (uint64_t)q * p.slot_bytes);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    if (q >= N) break;
                    const uint4 x = (q == r) ? own : val[j];
                    if (q == 0) acc = M::load(x);
                    else M::add(acc, x);
                }
            }
            store_output<T>(p.recv[r], base + v, p.count, M::store(acc));
        }
        if (!flag_barrier(p, s, tag + 1u, w, fail)) return false;  // buffers free again
    }
    return true;
}

template <typename T>
__global__ void __launch_bounds__(256) oneshot_barrier_kernel(const __grid_constant__ Params p) {
    __shared__ int fail;
    pdl_entry();
    if (threadIdx.x == 0) fail = 0;
    CtaState s = cta_prologue(p);
    s.skip = __syncthreads_or(s.skip) != 0;
    if (!s.skip) (void)oneshot_barrier_body<T>(p, s, &fail);
    cta_epilogue(p, s);
}

// Two-shot with barriers (the design the paper replaces, Sec. III-B, here for
// the two-shot of Sec. III-A): per step, plain stores of partition q of the
// chunk into window q's ReduceScatter slot [r]; an N-way flag barrier; the
// owner reduces its partition in rank order and stores the result into its
// own output and into every window's AllGather slot [r]; a second barrier;
// every rank copies the gathered partitions into its output.  CTA c of every
// rank handles the same positions u of every partition, so the per-CTA flag
// barriers order every exchange.  Reuse: a step's ReduceScatter slots are
// consumed before its second barrier, its AllGather slots before the next
// step's first barrier, after which alone they are written again.
template <typename T>
__device__ __forceinline__ bool twoshot_barrier_body(const Params& p, const CtaState& s, int* fail) {
    using M = VecMath<T>;
    const int N = p.nranks, r = s.rank;
    char* const rs_mine = window(p, r) + p.region_off;
    char* const ag_mine = window(p, r) + p.aux2_off;
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t tag = (uint32_t)(2ull * e);
        const uint32_t base = k * p.chunk_vecs;
        const uint32_t rem = min(p.chunk_vecs, p.nvec - base);  // vectors of this step
        const uint32_t pk = (rem + (uint32_t)N - 1) / (uint32_t)N;  // partition of this step
        const uint32_t u0 = (uint32_t)s.sub * p.per_cta;
        const uint32_t u1 = min(u0 + p.per_cta, pk);
        w.step = (int)k;
        // ReduceScatter: plain stores into the owners' windows
        if (!s.drop) {
#pragma unroll 1
            for (uint32_t u = u0 + threadIdx.x; u < u1; u += blockDim.x) {
#pragma unroll 1
                for (int q = 0; q < N; ++q) {
                    const uint32_t v = (uint32_t)q * pk + u;
                    if (q == r || v >= rem) continue;
                    st_relaxed_v4(window(p, q) + p.region_off + (uint64_t)r * p.slot_bytes + (uint64_t)u * kVecBytes,
                                  load_input<T>(p.send[r], base + v, p.count));
                }
            }
        }
        if (!flag_barrier(p, s, tag, w, fail)) return false;  // partitions delivered
        // reduce my partition in rank order; AllGather: plain stores to every window
#pragma unroll 1
        for (uint32_t u = u0 + threadIdx.x; u < u1; u += blockDim.x) {
            const uint32_t pos = (uint32_t)r * pk + u;
            if (pos >= rem) continue;
            typename M::Acc acc;
#pragma unroll 1
            for (int q = 0; q < N; ++q) {
                const uint4 x = q == r ? load_input<T>(p.send[r], base + pos, p.count)
                                       : ld_relaxed_v4(rs_mine + (uint64_t)q * p.slot_bytes + (uint64_t)u * kVecBytes);
                if (q == 0) acc = M::load(x);
                else M::add(acc, x);
            }
            const uint4 out = M::store(acc);
            store_output<T>(p.recv[r], base + pos, p.count, out);
            if (!s.drop) {
#pragma unroll 1
                for (int d = 0; d < N; ++d)
                    if (d != r)
                        st_relaxed_v4(window(p, d) + p.aux2_off + (uint64_t)r * p.slot_bytes + (uint64_t)u * kVecBytes,
                                      out);
            }
        }
        if (!flag_barrier(p, s, tag + 1u, w, fail)) return false;  // reduced partitions delivered
#pragma unroll 1
        for (uint32_t u = u0 + threadIdx.x; u < u1; u += blockDim.x) {
#pragma unroll 1
            for (int q = 0; q < N; ++q) {
                const uint32_t pos = (uint32_t)q * pk + u;
                if (q == r || pos >= rem) continue;
                store_output<T>(p.recv[r], base + pos, p.count,
                                ld_relaxed_v4(ag_mine + (uint64_t)q * p.slot_bytes + (uint64_t)u * kVecBytes));
            }
        }
    }
    return true;
}

template <typename T>
__global__ void __launch_bounds__(256) twoshot_barrier_kernel(const __grid_constant__ Params p) {
    __shared__ int fail;
    pdl_entry();
    if (threadIdx.x == 0) fail = 0;
    CtaState s = cta_prologue(p);
    s.skip = __syncthreads_or(s.skip) != 0;
    if (!s.skip) (void)twoshot_barrier_body<T>(p, s, &fail);
    cta_epilogue(p, s);
}

// Barrier latency (Fig. 3 analogue): N ranks x 1 CTA run `nsteps` flag
// barriers back to back; CTA 0 records %globaltimer after the first and after
// the last barrier in timing[0..1].
__global__ void __launch_bounds__(256) barrier_probe_kernel(const __grid_constant__ Params p) {
    __shared__ int fail;
    pdl_entry();
    if (threadIdx.x == 0) fail = 0;
    CtaState s = cta_prologue(p);
    s.skip = __syncthreads_or(s.skip) != 0;
    if (!s.skip) {
        Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, s.rank, 0);
        uint64_t t_first = 0;
#pragma unroll 1
        for (uint32_t k = 0; k < p.nsteps; ++k) {
            w.step = (int)k;
            if (!flag_barrier(p, s, (uint32_t)(2ull * (s.epoch + k)), w, &fail)) break;
            if (k == 0) t_first = globaltimer_ns();
        }
        if (blockIdx.x == 0 && threadIdx.x == 0 && p.timing != nullptr) {
            p.timing[0] = t_first;
            p.timing[1] = globaltimer_ns();
        }
    }
    const Params& q = p;
    if (!s.skip) {  // epoch bookkeeping as for any call; no per-CTA timing here
        __syncthreads();
        const uint64_t next_m1 = s.epoch + q.nsteps - 1ull;
        for (unsigned slot = blockIdx.x + threadIdx.x * gridDim.x; slot < (unsigned)q.epoch_slots;
             slot += blockDim.x * gridDim.x)
            st_relaxed_u64(&q.ctrl->epoch_m1[slot], next_m1);
    }
}

// ------------------------------------------ two-shot, double buffered ----
// Sec. III-A "Two-shot" (ReduceScatter then AllGather, both push) with
// sentinel synchronisation and the bidirectional double buffering of Sec. IV /
// Fig. 4.  Step k covers N partitions of `part` vectors; rank q owns
// partition q.  RS: every rank stores its part q into owner q's RS slot
// [parity][r].  Owner: polls the N-1 RS slots, reduces in rank order, stores
// the result into every peer's AG slot [parity][owner] and its own output.
// AG: every rank polls the N-1 AG slots and writes its output.
struct Split {
    uint32_t base;  // first vector of the step
    uint32_t part;  // vectors per partition in this step
    uint32_t rem;   // vectors left from `base` to the end of the message
    __device__ __forceinline__ uint32_t valid(int q) const {  // vectors of partition q
        const uint32_t lo = (uint32_t)q * part;
        return rem > lo ? min(part, rem - lo) : 0u;
    }
    __device__ __forceinline__ uint32_t vec(int q, uint32_t v) const { return base + (uint32_t)q * part + v; }
};

constexpr int kLoadParts = 8;  // partitions whose input vectors are loaded together

// The last step shrinks its partitions so the remaining vectors spread over
// all owners; positions stay a prefix of the full-step positions.
__device__ __forceinline__ Split split_step(const Params& p, uint32_t k) {
    Split sp;
    const uint32_t full = (uint32_t)p.nranks * p.chunk_vecs;
    sp.base = k * full;
    sp.rem = p.nvec - sp.base;
    sp.part = sp.rem >= full ? p.chunk_vecs : (sp.rem + (uint32_t)p.nranks - 1u) / (uint32_t)p.nranks;
    return sp;
}

// kDirect: the owner stores its reduced partition straight into every rank's
// output (the output buffers play the part of registered symmetric memory,
// Sec. II-B), so the AllGather needs no scratch, no poll and no reset: one
// synchronisation hop per step instead of two.  Outputs are complete when the
// kernel completes; nothing inside the kernel reads them.
//
// Shape (for bandwidth): a thread handles one position of the partitions at a
// time; the push issues the input loads of up to kLoadParts partitions, the
// receive phases the polls of up to kPollParts sources, before waiting for
// any of them.  The planner gives each thread about one position per step and
// as many co-resident CTAs as the occupancy allows, so a step keeps the whole
// GPU's loads in flight; the kernel is built for 4 CTAs of 128 threads per SM
// (at most 128 registers per thread: it needs about that many without
// spilling).
constexpr int kPollParts = 4;  // sources polled with loads in flight at once (two-shot)

// L2 policies of the two-shot: its scratch is written and read back within a
// step (keep it in L2), its inputs and outputs stream through once.
struct TwoshotHints {
    uint64_t keep, stream;
};

// ReduceScatter push of position v of this step: part q of my input ->
// owner q's RS slot [r], the inputs of kLoadParts partitions loaded together.
template <typename T>
__device__ __forceinline__ void twoshot_push(const Params& p, const Split sp, int r, uint32_t v, uint64_t par_off,
                                             TwoshotHints h) {
    constexpr int U = VecMath<T>::kUnitBytes;
    const int N = p.nranks;
    const uint64_t off = p.region_off + par_off + (uint64_t)r * p.slot_bytes + (uint64_t)v * kVecBytes;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += kLoadParts) {
        uint4 x[kLoadParts];
#pragma unroll
        for (int j = 0; j < kLoadParts; ++j) {
            const int q = q0 + j;
            if (q < N && q != r && v < sp.valid(q)) x[j] = load_input_hint<T>(p.send[r], sp.vec(q, v), p.count, h.stream);
        }
#pragma unroll
        for (int j = 0; j < kLoadParts; ++j) {
            const int q = q0 + j;
            if (q < N && q != r && v < sp.valid(q)) st_scratch_hint<U>(window(p, q) + off, x[j], h.keep);
        }
    }
}

// One poll of a two-shot scratch vector (sentinel).
template <typename T>
__device__ __forceinline__ bool twoshot_poll(const char* slot, uint64_t pol, uint4& out) {
    constexpr int U = VecMath<T>::kUnitBytes;
    out = ld_scratch_hint<U>(slot, pol);
    return sentinel_arrived<U>(out);
}

// Owner of position v: poll the N-1 RS slots (kPollParts sources in flight),
// add in rank order, push the sum to every peer's AG slot [r] (kDirect: into
// every peer's output), store my own output, then reset the consumed slots
// (plain stores: the next writer of a slot is ordered after this thread by
// the credit chain -- the fence of a later step, or the kernel boundary).
template <typename T, bool kDirect>
__device__ __forceinline__ bool twoshot_own(const Params& p, const Split sp, int r, bool drop, uint32_t v,
                                            uint64_t par_off, Waiter& w, TwoshotHints h) {
    using M = VecMath<T>;
    constexpr int U = M::kUnitBytes;
    const int N = p.nranks;
    const uint4 own = load_input_hint<T>(p.send[r], sp.vec(r, v), p.count, h.stream);
    char* const slot0 = window(p, r) + p.region_off + par_off + (uint64_t)v * kVecBytes;
    typename M::Acc acc;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += kPollParts) {
        uint4 val[kPollParts];
        bool ok[kPollParts];
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            ok[j] = true;
            if (q < N && q != r) ok[j] = twoshot_poll<T>(slot0 + (uint64_t)q * p.slot_bytes, h.keep, val[j]);
        }
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            while (!ok[j]) {
                if (waiter_expired(w)) return false;
                ok[j] = twoshot_poll<T>(slot0 + (uint64_t)q * p.slot_bytes, h.keep, val[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            if (q >= N) break;
            const uint4 x = (q == r) ? own : val[j];
            if (q == 0) acc = M::load(x);
            else M::add(acc, x);
        }
    }
    const uint4 red = M::store(acc);
    if (!drop) {
        if (kDirect) {
#pragma unroll 1
            for (int q = 0; q < N; ++q)
                if (q != r) store_output_hint<T>(p.recv[q], sp.vec(r, v), p.count, red, h.stream);
        } else {
            char* dst = p.win0 + p.aux_off + par_off + (uint64_t)r * p.slot_bytes + (uint64_t)v * kVecBytes;
#pragma unroll 1
            for (int q = 0; q < N; ++q, dst += p.stride)
                if (q != r) st_scratch_hint<U>(dst, red, h.keep);
        }
    }
    store_output_hint<T>(p.recv[r], sp.vec(r, v), p.count, red, h.stream);
#pragma unroll 1
    for (int q = 0; q < N; ++q)
        if (q != r) st_weak_v4_hint(slot0 + (uint64_t)q * p.slot_bytes, sentinel_vec(), h.keep);
    return true;
}

// AllGather receive of position v: the N-1 reduced partitions of the other
// owners (sources whose partition does not reach v are skipped), polled
// kPollParts at a time, stored into my output, the slots reset (plain stores,
// as in twoshot_own).
template <typename T>
__device__ __forceinline__ bool twoshot_gather(const Params& p, const Split sp, int r, uint32_t v, uint64_t par_off,
                                               Waiter& w, TwoshotHints h) {
    const int N = p.nranks;
    char* const slot0 = window(p, r) + p.aux_off + par_off + (uint64_t)v * kVecBytes;
#pragma unroll 1
    for (int q0 = 0; q0 < N; q0 += kPollParts) {
        uint4 val[kPollParts];
        bool ok[kPollParts];
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            ok[j] = true;
            if (q < N && q != r && v < sp.valid(q)) ok[j] = twoshot_poll<T>(slot0 + (uint64_t)q * p.slot_bytes, h.keep, val[j]);
        }
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            while (!ok[j]) {
                if (waiter_expired(w)) return false;
                ok[j] = twoshot_poll<T>(slot0 + (uint64_t)q * p.slot_bytes, h.keep, val[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPollParts; ++j) {
            const int q = q0 + j;
            if (q < N && q != r && v < sp.valid(q)) {
                store_output_hint<T>(p.recv[r], sp.vec(q, v), p.count, val[j], h.stream);
                st_weak_v4_hint(slot0 + (uint64_t)q * p.slot_bytes, sentinel_vec(), h.keep);
            }
        }
    }
    return true;
}

template <typename T, bool kDirect>
__device__ __forceinline__ bool twoshot_body(const Params& p, const CtaState& s) {
    const int r = s.rank;
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;
    const uint32_t pos1 = pos0 + p.per_cta;
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);
    const TwoshotHints h{l2_keep_policy(), l2_stream_policy()};

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint64_t par_off = (e & 1ull) * p.parity_bytes;
        const Split sp = split_step(p, k);
        const uint32_t end = min(pos1, sp.part);
        w.step = (int)k;
        if (k > 0 && p.nsteps > 2) fence_acq_rel_gpu();
        if (!s.drop) {
#pragma unroll 1
            for (uint32_t v = pos0 + threadIdx.x; v < end; v += blockDim.x) twoshot_push<T>(p, sp, r, v, par_off, h);
        }
        const uint32_t my_end = min(end, sp.valid(r));
#pragma unroll 1
        for (uint32_t v = pos0 + threadIdx.x; v < my_end; v += blockDim.x)
            if (!twoshot_own<T, kDirect>(p, sp, r, s.drop, v, par_off, w, h)) return false;
#pragma unroll 1
        for (uint32_t v = pos0 + threadIdx.x; !kDirect && v < end; v += blockDim.x)
            if (!twoshot_gather<T>(p, sp, r, v, par_off, w, h)) return false;
    }
    return true;
}

template <typename T, bool kDirect>
__global__ void __launch_bounds__(128, 4) twoshot_kernel(const __grid_constant__ Params p) {
    pdl_release_early();
    warm_params(p);
    pdl_wait();
    const CtaState s = cta_prologue(p, p.nsteps > 1);
    if (!s.skip) (void)twoshot_body<T, kDirect>(p, s);
    cta_epilogue(p, s);
}

// ------------------------------------------------ two-shot LL128 atomic ----
// Fig. 5: the ReduceScatter adds straight into the owner's destination lines
// with atomic additions and raises a per-line counter; the owner consumes a
// line when its counter shows every contribution (here: the N-1 peers, the
// owner adds its own part in registers), re-zeroes line and counter for the
// next use of the parity, and the AllGather pushes the result with epoch
// flags (LL encoding) to every peer.
//
// Single-GPU reading of the line atomicity the paper takes from NVLink: L2
// atomics are per element, so a contributor warp first issues all its
// red.add operations for a group of 32 vectors, synchronises the warp, and
// every lane issues fence.acq_rel.gpu before the counter increments (release);
// the owner's lane 0 reads the counter, fences (acquire) and synchronises the
// warp before the lanes read the lines.
template <typename T>
struct Acc128;
template <>
struct Acc128<float> {          // binary32 -> binary32 accumulators
    static constexpr int kRatio = 1;
    __device__ __forceinline__ static void red(char* dst, uint4 x) {
        red_add_v4f32(dst, __uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                      __uint_as_float(x.w));
    }
    __device__ __forceinline__ static uint4 finish(const char* src, uint4 own) {
        const uint4 a = ld_relaxed_v4(src);
        return make_uint4(__float_as_uint(__fadd_rn(__uint_as_float(a.x), __uint_as_float(own.x))),
                          __float_as_uint(__fadd_rn(__uint_as_float(a.y), __uint_as_float(own.y))),
                          __float_as_uint(__fadd_rn(__uint_as_float(a.z), __uint_as_float(own.z))),
                          __float_as_uint(__fadd_rn(__uint_as_float(a.w), __uint_as_float(own.w))));
    }
    __device__ __forceinline__ static void zero(char* src) { st_relaxed_v4(src, make_uint4(0, 0, 0, 0)); }
};
template <>
struct Acc128<__nv_bfloat16> {  // bfloat16 -> binary32 accumulators (2 x 16 B per vector)
    static constexpr int kRatio = 2;
    using VM = VecMath<__nv_bfloat16>;
    __device__ __forceinline__ static void red(char* dst, uint4 x) {
        red_add_v4f32(dst, VM::lo(x.x), VM::hi(x.x), VM::lo(x.y), VM::hi(x.y));
        red_add_v4f32(dst + 16, VM::lo(x.z), VM::hi(x.z), VM::lo(x.w), VM::hi(x.w));
    }
    __device__ __forceinline__ static uint4 finish(const char* src, uint4 own) {
        const uint4 a = ld_relaxed_v4(src);
        const uint4 b = ld_relaxed_v4(src + 16);
        const float f0 = __fadd_rn(__uint_as_float(a.x), VM::lo(own.x));
        const float f1 = __fadd_rn(__uint_as_float(a.y), VM::hi(own.x));
        const float f2 = __fadd_rn(__uint_as_float(a.z), VM::lo(own.y));
        const float f3 = __fadd_rn(__uint_as_float(a.w), VM::hi(own.y));
        const float f4 = __fadd_rn(__uint_as_float(b.x), VM::lo(own.z));
        const float f5 = __fadd_rn(__uint_as_float(b.y), VM::hi(own.z));
        const float f6 = __fadd_rn(__uint_as_float(b.z), VM::lo(own.w));
        const float f7 = __fadd_rn(__uint_as_float(b.w), VM::hi(own.w));
        return make_uint4(VM::pack(f0, f1), VM::pack(f2, f3), VM::pack(f4, f5), VM::pack(f6, f7));
    }
    __device__ __forceinline__ static void zero(char* src) {
        st_relaxed_v4(src, make_uint4(0, 0, 0, 0));
        st_relaxed_v4(src + 16, make_uint4(0, 0, 0, 0));
    }
};
template <>
struct Acc128<double> {         // binary64 -> binary64 accumulators
    static constexpr int kRatio = 1;
    using VM = VecMath<double>;
    __device__ __forceinline__ static void red(char* dst, uint4 x) {
        red_add_f64(dst, VM::d(x.x, x.y));
        red_add_f64(dst + 8, VM::d(x.z, x.w));
    }
    __device__ __forceinline__ static uint4 finish(const char* src, uint4 own) {
        uint64_t a, b;
        ld_relaxed_v2u64(src, a, b);
        const double d0 = __dadd_rn(__longlong_as_double((long long)a), VM::d(own.x, own.y));
        const double d1 = __dadd_rn(__longlong_as_double((long long)b), VM::d(own.z, own.w));
        return make_uint4((uint32_t)__double2loint(d0), (uint32_t)__double2hiint(d0),
                          (uint32_t)__double2loint(d1), (uint32_t)__double2hiint(d1));
    }
    __device__ __forceinline__ static void zero(char* src) { st_relaxed_v2u64(src, 0ull, 0ull); }
};

template <typename T>
__device__ __forceinline__ bool ll128_body(const Params& p, const CtaState& s) {
    using A = Acc128<T>;
    constexpr uint32_t kAccBytes = (uint32_t)kVecBytes * A::kRatio;
    const int N = p.nranks, r = s.rank;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t wbase = threadIdx.x - lane;               // first thread of this warp
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;       // per_cta is a multiple of 32
    const uint32_t pos1 = pos0 + p.per_cta;
    char* const mine = window(p, r);
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);
    const uint32_t target = (uint32_t)(N - 1);

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t ep = (uint32_t)e;
        const uint64_t par = e & 1ull;
        const Split sp = split_step(p, k);
        const uint32_t end = min(pos1, sp.part);
        w.step = (int)k;
        if (k > 0 && p.nsteps > 2) fence_acq_rel_gpu();

        // ReduceScatter: atomic adds into each owner's accumulators.  Loop
        // bounds use the warp's first position, so they are warp-uniform.
        if (!s.drop) {
#pragma unroll 1
            for (uint32_t g0 = pos0 + wbase; g0 < end; g0 += blockDim.x) {
                const uint32_t v = g0 + lane;
                const uint64_t off = p.region_off + par * p.parity_bytes + (uint64_t)v * kAccBytes;
#pragma unroll 1
                for (int q0 = 0; q0 < N; q0 += kLoadParts) {
                    uint4 x[kLoadParts];
#pragma unroll
                    for (int j = 0; j < kLoadParts; ++j) {
                        const int q = q0 + j;
                        if (q < N && q != r && v < sp.valid(q)) x[j] = load_input<T>(p.send[r], sp.vec(q, v), p.count);
                    }
#pragma unroll
                    for (int j = 0; j < kLoadParts; ++j) {
                        const int q = q0 + j;
                        if (q < N && q != r && v < sp.valid(q)) A::red(window(p, q) + off, x[j]);
                    }
                }
            }
            __syncwarp();
            fence_acq_rel_gpu();  // release: this warp's adds before its counter increments
#pragma unroll 1
            for (uint32_t g0 = pos0 + wbase; g0 < end; g0 += blockDim.x) {
                const uint64_t coff = p.aux_off + par * p.aux_parity_bytes + (uint64_t)(g0 / kGroupVecs) * 4;
#pragma unroll 1
                for (int q = (int)lane; q < N; q += 32) {
                    if (q == r || g0 >= sp.valid(q)) continue;
                    red_add_u32(window(p, q) + coff, 1u);
                }
            }
        }
        // Owner: wait for each group's counter, consume, re-zero, AllGather push.
        const uint32_t my_end = min(end, sp.valid(r));
#pragma unroll 1
        for (uint32_t g0 = pos0 + wbase; g0 < my_end; g0 += blockDim.x) {
            char* const cnt = mine + p.aux_off + par * p.aux_parity_bytes + (uint64_t)(g0 / kGroupVecs) * 4;
            int give_up = 0;
            if (lane == 0) {
                while (ld_relaxed_u32(cnt) != target) {
                    if (waiter_expired(w)) { give_up = 1; break; }
                }
                fence_acq_rel_gpu();  // acquire: the counter before the lines
            }
            if (__shfl_sync(0xFFFFFFFFu, give_up, 0)) return false;
            __syncwarp();
            const uint32_t v = g0 + lane;
            if (v < my_end) {
                char* const acc = mine + p.region_off + par * p.parity_bytes + (uint64_t)v * kAccBytes;
                const uint4 own = load_input<T>(p.send[r], sp.vec(r, v), p.count);
                const uint4 red = A::finish(acc, own);
                A::zero(acc);
                if (!s.drop) {
                    char* dst = p.win0 + p.aux2_off + par * p.aux2_parity_bytes + (uint64_t)r * p.aux2_slot_bytes +
                                (uint64_t)v * (2 * kVecBytes);
#pragma unroll 1
                    for (int q = 0; q < N; ++q, dst += p.stride) {
                        if (q != r) ll_store(dst, red, ep);
                    }
                }
                store_output<T>(p.recv[r], sp.vec(r, v), p.count, red);
            }
            __syncwarp();
            if (lane == 0) st_relaxed_u32(cnt, 0u);
        }
        // AllGather receive (LL polls), per lane; the warp leaves together.
        int failed = 0;
#pragma unroll 1
        for (uint32_t g0 = pos0 + wbase; g0 < end; g0 += blockDim.x) {
            const uint32_t v = g0 + lane;
            if (failed || v >= end) continue;
            char* const slot0 = mine + p.aux2_off + par * p.aux2_parity_bytes + (uint64_t)v * (2 * kVecBytes);
#pragma unroll 1
            for (int q0 = 0; q0 < N; q0 += kBatch) {
                uint4 val[kBatch];
                bool ok[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    ok[j] = true;
                    if (q < N && q != r && v < sp.valid(q))
                        ok[j] = ll_load(slot0 + (uint64_t)q * p.aux2_slot_bytes, ep, val[j]);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    while (!ok[j]) {
                        if (waiter_expired(w)) { failed = 1; break; }
                        ok[j] = ll_load(slot0 + (uint64_t)q * p.aux2_slot_bytes, ep, val[j]);
                    }
                    if (failed) break;
                }
                if (failed) break;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int q = q0 + j;
                    if (q < N && q != r && v < sp.valid(q))
                        store_output<T>(p.recv[r], sp.vec(q, v), p.count, val[j]);
                }
            }
        }
        if (__any_sync(0xFFFFFFFFu, failed)) return false;
    }
    return true;
}

// Wide variant for many ranks: the threads of a CTA split the (owner q,
// position v) items of the ReduceScatter's atomic adds and of the AllGather's
// polls, so a small partition no longer leaves one thread walking the N-1
// owners in order.  The counter of a group (32 positions, inside one CTA) is
// incremented once per contributing rank after a CTA-wide release: every
// thread fences its adds, the CTA meets, then one thread per (owner, group)
// increments.  Same owner phase and results as ll128_body.
template <typename T>
__device__ __forceinline__ bool ll128_wide_body(const Params& p, const CtaState& s) {
    using A = Acc128<T>;
    constexpr uint32_t kAccBytes = (uint32_t)kVecBytes * A::kRatio;
    const int N = p.nranks, r = s.rank;
    const uint32_t nt = blockDim.x;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t wbase = threadIdx.x - lane;
    const uint32_t pos0 = (uint32_t)s.sub * p.per_cta;  // per_cta is a multiple of 32
    const uint32_t pos1 = pos0 + p.per_cta;
    char* const mine = window(p, r);
    Waiter w = make_waiter(s.t_start, p.timeout_ns, p.ctrl, r, 0);
    const uint32_t target = (uint32_t)(N - 1);

#pragma unroll 1
    for (uint32_t k = 0; k < p.nsteps; ++k) {
        const uint64_t e = s.epoch + k;
        const uint32_t ep = (uint32_t)e;
        const uint64_t par = e & 1ull;
        const Split sp = split_step(p, k);
        const uint32_t end = min(pos1, sp.part);
        const uint32_t np = end > pos0 ? end - pos0 : 0u;  // this CTA's positions in this step
        const uint32_t items = (uint32_t)N * np;           // (owner q, position) pairs
        w.step = (int)k;
        if (k > 0 && p.nsteps > 2) fence_acq_rel_gpu();

        // ReduceScatter: atomic adds, one item per thread and batch
        if (!s.drop) {
#pragma unroll 1
            for (uint32_t b0 = 0; b0 < items; b0 += nt * (uint32_t)kLoadParts) {
                uint4 x[kLoadParts];
#pragma unroll
                for (int j = 0; j < kLoadParts; ++j) {
                    const uint32_t it = b0 + threadIdx.x + (uint32_t)j * nt;
                    if (it >= items) continue;
                    const int q = (int)(it / np);
                    const uint32_t v = pos0 + (it - (uint32_t)q * np);
                    if (q != r && v < sp.valid(q)) x[j] = load_input<T>(p.send[r], sp.vec(q, v), p.count);
                }
#pragma unroll
                for (int j = 0; j < kLoadParts; ++j) {
                    const uint32_t it = b0 + threadIdx.x + (uint32_t)j * nt;
                    if (it >= items) continue;
                    const int q = (int)(it / np);
                    const uint32_t v = pos0 + (it - (uint32_t)q * np);
                    if (q != r && v < sp.valid(q))
                        A::red(window(p, q) + p.region_off + par * p.parity_bytes + (uint64_t)v * kAccBytes, x[j]);
                }
            }
            fence_acq_rel_gpu();  // release: this thread's adds before any counter increment
            __syncthreads();
            const uint32_t g_first = pos0 / kGroupVecs;
            const uint32_t ng = np == 0 ? 0u : (end - 1) / kGroupVecs - g_first + 1;
#pragma unroll 1
            for (uint32_t it = threadIdx.x; it < (uint32_t)N * ng; it += nt) {
                const int q = (int)(it / ng);
                const uint32_t g = g_first + (it - (uint32_t)q * ng);
                if (q == r || g * kGroupVecs >= sp.valid(q)) continue;
                red_add_u32(window(p, q) + p.aux_off + par * p.aux_parity_bytes + (uint64_t)g * 4, 1u);
            }
        }
        // Owner: per group (a warp), wait for the counter, consume, re-zero,
        // AllGather push.  A warp that gives up stops; the CTA decides below.
        int failed = 0;
        const uint32_t my_end = min(end, sp.valid(r));
#pragma unroll 1
        for (uint32_t g0 = pos0 + wbase; g0 < my_end; g0 += nt) {
            char* const cnt = mine + p.aux_off + par * p.aux_parity_bytes + (uint64_t)(g0 / kGroupVecs) * 4;
            int give_up = 0;
            if (lane == 0) {
                while (ld_relaxed_u32(cnt) != target) {
                    if (waiter_expired(w)) { give_up = 1; break; }
                }
                fence_acq_rel_gpu();  // acquire: the counter before the lines
            }
            if (__shfl_sync(0xFFFFFFFFu, give_up, 0)) {
                failed = 1;
                break;
            }
            __syncwarp();
            const uint32_t v = g0 + lane;
            if (v < my_end) {
                char* const acc = mine + p.region_off + par * p.parity_bytes + (uint64_t)v * kAccBytes;
                const uint4 own = load_input<T>(p.send[r], sp.vec(r, v), p.count);
                const uint4 red = A::finish(acc, own);
                A::zero(acc);
                if (!s.drop) {
                    char* dst = p.win0 + p.aux2_off + par * p.aux2_parity_bytes + (uint64_t)r * p.aux2_slot_bytes +
                                (uint64_t)v * (2 * kVecBytes);
#pragma unroll 1
                    for (int q = 0; q < N; ++q, dst += p.stride) {
                        if (q != r) ll_store(dst, red, ep);
                    }
                }
                store_output<T>(p.recv[r], sp.vec(r, v), p.count, red);
            }
            __syncwarp();
            if (lane == 0) st_relaxed_u32(cnt, 0u);
        }
        if (__syncthreads_or(failed)) return false;
        // AllGather receive: (owner q, position v) items spread over the CTA
#pragma unroll 1
        for (uint32_t b0 = 0; b0 < items && !failed; b0 += nt * (uint32_t)kBatch) {
            uint4 val[kBatch];
            bool ok[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const uint32_t it = b0 + threadIdx.x + (uint32_t)j * nt;
                ok[j] = true;
                if (it >= items) continue;
                const int q = (int)(it / np);
                const uint32_t v = pos0 + (it - (uint32_t)q * np);
                if (q != r && v < sp.valid(q))
                    ok[j] = ll_load(mine + p.aux2_off + par * p.aux2_parity_bytes + (uint64_t)q * p.aux2_slot_bytes +
                                        (uint64_t)v * (2 * kVecBytes),
                                    ep, val[j]);
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const uint32_t it = b0 + threadIdx.x + (uint32_t)j * nt;
                if (it >= items) continue;
                const int q = (int)(it / np);
                const uint32_t v = pos0 + (it - (uint32_t)q * np);
                if (q == r || v >= sp.valid(q)) continue;
                const char* const slot = mine + p.aux2_off + par * p.aux2_parity_bytes +
                                         (uint64_t)q * p.aux2_slot_bytes + (uint64_t)v * (2 * kVecBytes);
                while (!ok[j] && !failed) {
                    if (waiter_expired(w)) failed = 1;
                    else ok[j] = ll_load(slot, ep, val[j]);
                }
                if (ok[j]) store_output<T>(p.recv[r], sp.vec(q, v), p.count, val[j]);
            }
        }
        if (__syncthreads_or(failed)) return false;
    }
    return true;
}

template <typename T>
__global__ void __launch_bounds__(256) ll128_wide_kernel(const __grid_constant__ Params p) {
    pdl_release_early();
    warm_params(p);
    pdl_wait();
    CtaState s = cta_prologue(p);
    s.skip = __syncthreads_or(s.skip) != 0;  // CTA-wide syncs follow: skip must be CTA-uniform
    if (!s.skip) (void)ll128_wide_body<T>(p, s);
    cta_epilogue(p, s);
}

template <typename T>
__global__ void __launch_bounds__(256) ll128_kernel(const __grid_constant__ Params p) {
    pdl_release_early();
    warm_params(p);
    pdl_wait();
    CtaState s = cta_prologue(p);
    s.skip = __any_sync(0xFFFFFFFFu, s.skip) != 0;  // warp syncs follow: skip must be warp-uniform
    if (!s.skip) (void)ll128_body<T>(p, s);
    cta_epilogue(p, s);
}

// ---------------------------------------------------------- initialiser ----
// Fills every window region with its idle pattern (sentinel regions all-ones,
// LL flags / accumulators / counters zero) and resets the control block.
struct FillJob {
    uint64_t off;    // offset inside a window
    uint64_t bytes;  // multiple of 16
    uint32_t value;  // 32-bit fill pattern
};
struct InitParams {
    char* win0;
    Ctrl* ctrl;
    uint64_t stride;
    int nranks;
    int njobs;
    FillJob job[6];
};

__global__ void init_kernel(const __grid_constant__ InitParams ip) {
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            ip.ctrl->status = 0u;
            ip.ctrl->err_rank = -1;
            ip.ctrl->err_step = -1;
            ip.ctrl->scrub_arrive = 0u;
            ip.ctrl->scrub_gen = 0u;
        }
        for (int i = threadIdx.x; i < kEpochSlots; i += blockDim.x) ip.ctrl->epoch_m1[i] = 0ull;  // epoch 1
    }
    for (int r = 0; r < ip.nranks; ++r) {
        for (int j = 0; j < ip.njobs; ++j) {
            const FillJob& f = ip.job[j];
            const uint4 v = make_uint4(f.value, f.value, f.value, f.value);
            uint4* dst = (uint4*)(ip.win0 + (uint64_t)r * ip.stride + f.off);
            for (uint64_t i = tid; i < f.bytes / 16; i += nthreads) dst[i] = v;
        }
    }
}

// --------------------------------------------------------- host launch ----
template <typename T>
static const void* kernel_for(int kind, bool trace) {
    switch (kind) {
        case kKindOneshotLL:
            return trace ? (const void*)oneshot_kernel<T, true, true> : (const void*)oneshot_kernel<T, true, false>;
        case kKindOneshotSentinel:
            return trace ? (const void*)oneshot_kernel<T, false, true> : (const void*)oneshot_kernel<T, false, false>;
        case kKindTwoshot: return (const void*)twoshot_kernel<T, false>;
        case kKindTwoshotDirect: return (const void*)twoshot_kernel<T, true>;
        case kKindLL128: return (const void*)ll128_kernel<T>;
        case kKindLL128Wide: return (const void*)ll128_wide_kernel<T>;
        case kKindOneshotLLWide: return (const void*)oneshot_wide_kernel<T, true>;
        case kKindOneshotSentinelWide: return (const void*)oneshot_wide_kernel<T, false>;
        case kKindOneshotBarrier: return (const void*)oneshot_barrier_kernel<T>;
        case kKindTwoshotBarrier: return (const void*)twoshot_barrier_kernel<T>;
        case kKindBarrierProbe: return (const void*)barrier_probe_kernel;
    }
    return nullptr;
}

// trace: the one-shot's variant with trace points (a trace buffer is set).
static const void* kernel_for(rra_dtype_t dtype, int kind, bool trace = false) {
    switch (dtype) {
        case RRA_FP32: return kernel_for<float>(kind, trace);
        case RRA_BF16: return kernel_for<__nv_bfloat16>(kind, trace);
        case RRA_FP64: return kernel_for<double>(kind, trace);
    }
    return nullptr;
}

cudaError_t occupancy(rra_dtype_t dtype, int kind, int threads, int* blocks_per_sm) {
    const void* k = kernel_for(dtype, kind);
    if (k == nullptr) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, threads, 0);
}

// Whether a one-shot launch of `grid` CTAs, one per rank, runs as one
// thread-block cluster.  The CTAs of a cluster are scheduled together on one
// GPC, so every rank's pushes and polls stay on one die of the GPU: at 128 B
// per rank this measured 5-17 % less in-kernel time at 4-16 ranks (none at 2,
// none for the two-shot or LL128 kernels, which are left as they are), and
// the co-scheduling of a cluster also makes every CTA resident together.
// Only calls with one CTA per rank and 2-16 CTAs qualify; the answer for
// each (kernel, grid, threads) is asked of cudaOccupancyMaxActiveClusters
// once and kept.
static bool one_cluster(const void* k, int kind, const Params& p, unsigned grid, int threads) {
    if (kind != kKindOneshotLL && kind != kKindOneshotSentinel && kind != kKindOneshotLLWide &&
        kind != kKindOneshotSentinelWide)
        return false;
    if (p.ctas_per_rank != 1 || grid < 2 || grid > 16) return false;
    struct Fit {
        const void* k;
        unsigned grid;
        int threads;
        bool fits;
    };
    static std::mutex mu;
    static Fit fit[96];
    static int nfit = 0;
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < nfit; ++i)
        if (fit[i].k == k && fit[i].grid == grid && fit[i].threads == threads) return fit[i].fits;
    bool fits = false;
    if (grid <= 8 || cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3((unsigned)threads);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = grid;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        fits = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) == cudaSuccess && clusters >= 1;
    }
    cudaGetLastError();
    if (nfit < (int)(sizeof(fit) / sizeof(fit[0]))) fit[nfit++] = Fit{k, grid, threads, fits};
    return fits;
}

cudaError_t launch_allreduce(const Params& p, rra_dtype_t dtype, int kind, int threads, cudaStream_t stream,
                             bool cooperative, bool pdl) {
    const void* k = kernel_for(dtype, kind, p.trace != nullptr);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nranks * p.ctas_per_rank));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (one_cluster(k, kind, p, cfg.gridDim.x, threads)) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cfg.gridDim.x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
        cooperative = false;  // a cluster's CTAs are resident together
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
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

cudaError_t launch_init(char* base, size_t total, const rra_layout_t& lay, int nranks,
                        cudaStream_t stream) {
    (void)total;
    InitParams ip = {};
    ip.ctrl = (Ctrl*)base;
    ip.win0 = base + lay.ctrl_bytes;
    ip.stride = lay.window_stride;
    ip.nranks = nranks;
    uint64_t off = 0;
    int j = 0;
    // Region order inside a window: LL slots, barrier flags, sentinel one-shot,
    // two-shot (RS+AG), LL128 (accumulators + counters + LL AllGather),
    // barrier-baseline data.  Must match the planner.
    ip.job[j++] = FillJob{off, lay.ll_bytes + lay.bf_bytes, 0u};  off += lay.ll_bytes + lay.bf_bytes;
    ip.job[j++] = FillJob{off, lay.os_bytes, 0xFFFFFFFFu};        off += lay.os_bytes;
    ip.job[j++] = FillJob{off, lay.ts_bytes, 0xFFFFFFFFu};        off += lay.ts_bytes;
    ip.job[j++] = FillJob{off, lay.la_bytes, 0u};                 off += lay.la_bytes;
    ip.job[j++] = FillJob{off, lay.bd_bytes, 0u};                 off += lay.bd_bytes;
    ip.njobs = j;
    init_kernel<<<1024, 256, 0, stream>>>(ip);
    return cudaGetLastError();
}

}  // namespace rra
