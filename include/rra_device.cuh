/*
 * rra_device.cuh -- device-side low-latency communication API for writing
 * custom collective kernels on one GB300 (header only, sm_103a).
 *
 * "Every Microsecond Matters: Achieving Near Speed-of-Light Latency in GPU
 * Collectives" (Abstract; Sec. I, contributions; Fig. 6-9) puts a small
 * device-side API under its kernels so that custom collectives can be
 * written with the same barrier-free synchronisation: a per-CTA buffer
 * whose region alternates between two sub-buffers from one epoch to the
 * next (Fig. 7), send() into a given peer's slot (Fig. 8), a push to all
 * peers, used by the one-shot AllReduce (Fig. 9), a receive that waits on
 * the arrival of the data itself, and advanceEpoch() to switch sub-buffers.
 *
 * Restated for one GB300: the virtual ranks of a team are the CTAs of one
 * thread-block cluster (CTA r of the cluster acts as rank r; up to 16
 * ranks), and a rank's buffer is a window in its own shared memory.  A send
 * is an st.async into the peer's window; it also completes the peer's
 * mbarrier transaction count, so the receiver waits on its own mbarrier and
 * the arrival of the bytes is the signal (the in-line LL flag of the pages
 * becomes the mbarrier's byte count).  Nothing persists between launches.
 *
 * Window layout, in the calling CTA's shared memory (16-byte aligned):
 *     window[sub][p][i],  sub = epoch & 1,  p < nranks,  i < slot_vecs
 * slot [p] of a sub-buffer receives what rank p sends in that epoch.
 * Size: 2 * nranks * slot_vecs * 16 bytes.
 *
 * Use (every thread of every CTA of the cluster calls every member, in the
 * same order, unless a comment says otherwise):
 *     __shared__ __align__(8) uint64_t bars[2];
 *     extern __shared__ __align__(16) uint4 window[];
 *     rra_dev::Team t;
 *     t.setup(window, bars, slot_vecs, bytes_expected_in_epoch_0);
 *     ...                       // may wait for the previous kernel here
 *     t.ready();                // peers' windows exist; sends allowed
 *     t.send(peer, i, v) / t.bcast(i, v) / t.put(i, v)   (any thread)
 *     t.bulk_send(peer, i, src, n) / t.bulk_bcast(i, src, n, ranks)  (one thread)
 *     if (!t.wait(deadline)) { ... gave up ... }
 *     x = t.recv(p, i);         (any thread)
 *     t.advance_epoch(bytes_expected_next);   // next sub-buffer
 *     ...
 *     t.sent();                 // after the last send of the kernel
 *     t.finish();               // last call before the CTA exits
 *
 * Reuse rule (the pages' double buffering, in which having received from a
 * peer is what allows the next send to it).  A sub-buffer is written again
 * two epochs later.  That is safe
 * when, in every epoch, each rank receives something from every peer that
 * will write into its window two epochs later (as in every AllReduce-like
 * exchange): a peer's epoch e+2 send then follows its epoch e+1 receive,
 * which follows this CTA's epoch e+1 send, which advance_epoch() orders
 * after this CTA's reads of epoch e.
 *
 * Bulk sends (bulk_send / bulk_bcast) move whole runs of vectors from
 * global memory into the windows by the TMA engine (cp.async.bulk with
 * cluster multicast), without passing through registers; the copy
 * completes each destination's mbarrier like an st.async.  A CTA that
 * bulk-sends calls sent() only after its last wait(): finish() then also
 * means that every copy into every window of the team has landed.
 * Source rule: a bulk send's source range must lie entirely in device
 * memory of the GPU the kernel runs on -- not host memory (pinned, mapped
 * or managed), not another GPU's memory reached through peer access -- and
 * bulk sends belong only in kernels of a process that drives this one GPU
 * alone.  The caller checks this on the host before choosing a kernel with
 * bulk sends (librra does so with cudaPointerGetAttributes, and otherwise
 * launches its st.async variant); send() and bcast() have no such rule.
 *
 * Every wait is bounded by a %globaltimer deadline: a rank that never
 * sends makes its receivers return false from wait(), never hang.
 */
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rra_dev {
namespace detail {

__device__ __forceinline__ uint32_t ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint32_t map_to(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void arm(uint32_t bar, uint32_t bytes) {
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;" : "=l"(state) : "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
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

}  // namespace detail

class Team {
  public:
    // Thread 0 initialises both mbarriers and arms epoch 0 with the bytes
    // this CTA will receive in it; every thread then arrives (relaxed) on the
    // cluster barrier.  Touches no global memory, so a kernel may call it
    // before waiting for the previous kernel (griddepcontrol.wait).
    __device__ void setup(uint4* window, uint64_t* bars, uint32_t slot_vecs, uint32_t expect_bytes) {
        rank_ = detail::ctarank();
        nranks_ = detail::nctarank();
        slot_vecs_ = slot_vecs;
        epoch_ = 0;
        window_ = window;
        win_s_ = detail::smem_addr(window);
        bar_s_ = detail::smem_addr(bars);
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" : : "r"(bar_s_) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" : : "r"(bar_s_ + 8u) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            detail::arm(bar_s_, expect_bytes);
        }
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    }

    // Completes the cluster barrier begun in setup(): every peer's window
    // and mbarriers exist.  Call once, before the first send.
    __device__ void ready() const { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

    __device__ uint32_t rank() const { return rank_; }
    __device__ uint32_t nranks() const { return nranks_; }
    __device__ uint32_t epoch() const { return epoch_; }

    // Any thread: write v into vector i of this rank's slot in `peer`'s
    // current sub-buffer (peer != rank()).  Counts 16 bytes toward the
    // peer's expectation for this epoch.
    __device__ void send(uint32_t peer, uint32_t i, uint4 v) const {
        const uint32_t off = ((sub() * nranks_ + rank_) * slot_vecs_ + i) * 16u;
        const uint32_t dst = detail::map_to(win_s_ + off, peer);
        const uint32_t bar = detail::map_to(bar_s_ + 8u * sub(), peer);
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];"
                     :
                     : "r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                     : "memory");
    }

    // Any thread: send v to every peer (not to itself; see put()).
    __device__ void bcast(uint32_t i, uint4 v) const {
        for (uint32_t k = 1; k < nranks_; ++k) send(rank_ + k < nranks_ ? rank_ + k : rank_ + k - nranks_, i, v);
    }
    // One thread: copy nvec > 0 vectors from global memory at src (16-byte
    // aligned) into vectors i .. i + nvec - 1 of this rank's slot in the
    // current sub-buffer of every rank whose bit is set in `ranks` (this
    // rank's own bit included if wanted), by one bulk copy with cluster
    // multicast.  Counts nvec * 16 bytes toward each destination's
    // expectation for this epoch -- this rank's own slot too, unlike put().
    // src must stay unchanged until every destination has waited, and
    // [src, src + 16 nvec) must be device memory of this GPU (the source
    // rule above).
    __device__ void bulk_bcast(uint32_t i, const void* src, uint32_t nvec, uint32_t ranks) const {
        const uint32_t off = ((sub() * nranks_ + rank_) * slot_vecs_ + i) * 16u;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1], %2, "
            "[%3], %4;"
            :
            : "r"(win_s_ + off), "l"(src), "r"(nvec * 16u), "r"(bar_s_ + 8u * sub()), "h"((uint16_t)ranks)
            : "memory");
    }
    // One thread: bulk_bcast() to one rank (which may be this rank).
    __device__ void bulk_send(uint32_t peer, uint32_t i, const void* src, uint32_t nvec) const {
        bulk_bcast(i, src, nvec, 1u << peer);
    }

    // Any thread: write v into this rank's own slot of its current
    // sub-buffer (a local store; counts toward no expectation).
    __device__ void put(uint32_t i, uint4 v) const { window_[(sub() * nranks_ + rank_) * slot_vecs_ + i] = v; }

    // Every thread: wait until the bytes expected for this epoch have
    // arrived, or until %globaltimer passes deadline_ns.  Returns the same
    // value in every thread of the CTA (true = all arrived) and makes the
    // CTA's own put()s visible to all its threads.
    __device__ bool wait(uint64_t deadline_ns) const {
        const uint32_t bar = bar_s_ + 8u * sub();
        const uint32_t parity = (epoch_ >> 1) & 1u;
        int ok = 1;
        uint32_t spins = 0;
        while (!detail::try_wait(bar, parity)) {
            if ((++spins & 63u) == 0u && detail::now_ns() > deadline_ns) {
                ok = 0;
                break;
            }
        }
        return __syncthreads_and(ok) != 0;
    }

    // Any thread, after wait(): vector i of slot [p] of the current sub-buffer.
    __device__ uint4 recv(uint32_t p, uint32_t i) const { return window_[(sub() * nranks_ + p) * slot_vecs_ + i]; }

    // Every thread: end this epoch (all reads of the current sub-buffer done)
    // and arm the next one with the bytes this CTA will receive in it.  The
    // proxy fence orders this CTA's reads before later bulk copies into the
    // same sub-buffer.
    __device__ void advance_epoch(uint32_t expect_bytes) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        ++epoch_;
        if (threadIdx.x == 0) detail::arm(bar_s_ + 8u * sub(), expect_bytes);
    }

    // Every thread, after the kernel's last send: arrive (relaxed) on the
    // cluster barrier that finish() completes.
    __device__ void sent() const { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }

    // Every thread, last: wait until every peer has issued its sends into
    // this CTA's window, so that the window outlives them.
    __device__ void finish() const { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

  private:
    __device__ uint32_t sub() const { return epoch_ & 1u; }

    uint4* window_;
    uint32_t win_s_, bar_s_;
    uint32_t rank_, nranks_, slot_vecs_, epoch_;
};

}  // namespace rra_dev
