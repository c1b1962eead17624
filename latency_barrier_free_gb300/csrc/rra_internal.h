// rra_internal.h -- definitions shared by the host library and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "rra.h"

namespace rra {

constexpr int kMaxRanks = RRA_MAX_RANKS;
constexpr int kVecBytes = 16;          // every transfer unit is one 16-byte vector
constexpr int kEpochSlots = 1024;      // largest grid a communicator may launch
constexpr int kGroupVecs = 32;         // LL128-atomic: vectors per completion counter (one warp)
constexpr size_t kRegionAlign = 4096;
constexpr uint64_t kMaxMessageBytes = (1ull << 36) - 16;  // 16-byte vector indices fit in 32 bits
// LL flags are the low 32 bits of the epoch.  When a call's epochs would cross
// a multiple of kScrubPeriod, all LL flag regions are zeroed and the epoch
// restarts one past that multiple, so every live flag value is unique.
constexpr uint64_t kScrubPeriod = 1ull << 31;

// Control block at the start of the allocation (before window 0).  All-zero
// bytes (with all-zero windows: LL flags 0, counters 0) are the idle state:
// status 0, epoch 1.
struct Ctrl {
    uint32_t status;     // rra_status_t of the first device-side error; 0 = none
    int32_t err_rank;    // virtual rank that recorded it
    int32_t err_step;    // chunk step of the call in which it was recorded
    uint32_t scrub_arrive;  // LL flag scrub: CTAs arrived at the grid barrier
    uint32_t scrub_gen;     // LL flag scrub: completed scrubs (barrier generation)
    uint32_t* host_status;  // device address of a pinned host word that mirrors `status`
                            // (written with it on the first error), or null
    uint32_t reserved[56];
    // Every CTA slot holds the same value: the epoch of the next step, minus
    // one (so that zero is epoch 1).  CTA b of a call with G CTAs reads slot b
    // at entry and writes epoch + steps - 1 to every slot b' = b (mod G); each
    // slot has exactly one reader/writer per call, and all slots stay equal
    // whatever grid a later call uses.
    uint64_t epoch_m1[kEpochSlots];
};

// Kernel parameters, passed by value (one launch = one call).
struct Params {
    const void* send[kMaxRanks];
    void* recv[kMaxRanks];
    char* win0;            // window 0 (window r = win0 + r * stride)
    Ctrl* ctrl;
    uint64_t* timing;      // optional: (start, end) %globaltimer per CTA
    uint64_t* trace;       // optional: kTracePoints %globaltimer stamps per CTA (one-shot)
    uint64_t stride;       // bytes between windows
    uint64_t count;        // elements per rank
    uint64_t timeout_ns;   // limit of every wait
    uint64_t region_off;   // offset of the algorithm's region inside a window
    uint64_t slot_bytes;   // bytes of one (parity, source) slot
    uint64_t parity_bytes; // bytes of one parity (all sources)
    uint64_t aux_off;      // two-shot: AllGather region; LL128: counters
    uint64_t aux2_off;     // LL128: LL-encoded AllGather slots
    uint64_t aux_parity_bytes;   // LL128: bytes of one parity of counters
    uint64_t aux2_slot_bytes;    // LL128: bytes of one AllGather slot
    uint64_t aux2_parity_bytes;  // LL128: bytes of one AllGather parity
    uint64_t ll_off, ll_bytes;        // LL flag regions of a window (one-shot LL slots,
    uint64_t llag_off, llag_bytes;    // LL128 AllGather slots), zeroed by the epoch scrub
    uint32_t nvec;         // 16-byte vectors per rank = ceil(count / elems per vector)
    uint32_t chunk_vecs;   // one-shot: vectors per rank per full step;
                           // two-shot/LL128: vectors per partition per full step
    uint32_t per_cta;      // vectors per CTA per step (the same in every step)
    uint32_t nsteps;
    int32_t nranks;
    int32_t ctas_per_rank;
    int32_t epoch_slots;   // number of epoch slots to keep equal
    int32_t root;          // Broadcast / Reduce: the root rank
    int32_t drop_rank;     // injected fault: rank whose stores to peers are skipped; -1 = none
    int32_t scrub_ranks;   // windows the epoch scrub zeroes (0: nranks)
};

// Kernel kinds: the algorithms (same values as rra_algo_t) plus the wide
// one-shot and LL128-atomic variants that split a position's sources over
// threads.
enum KernelKind {
    kKindOneshotLL = RRA_ONESHOT_LL,
    kKindOneshotSentinel = RRA_ONESHOT_SENTINEL,
    kKindTwoshot = RRA_TWOSHOT_DBUF,
    kKindLL128 = RRA_LL128_ATOMIC,
    kKindOneshotBarrier = RRA_ONESHOT_BARRIER,
    kKindTwoshotDirect = RRA_TWOSHOT_DIRECT,
    kKindOneshotLLWide = 6,
    kKindOneshotSentinelWide = 7,
    kKindBarrierProbe = 8,
    kKindTwoshotBarrier = RRA_TWOSHOT_BARRIER,
    kKindLL128Wide = 10,
    kNumKinds = 11
};
constexpr int kBarrierCtas = 64;  // CTAs per rank of the barrier baseline (flag slots per window)
constexpr int kWideStageVecs = 3072;  // wide one-shot: shared-memory stage, in 16-byte vectors
constexpr int kTracePoints = 6;       // start, control words read, pushed, polled, stored, end
constexpr size_t kClusterStageBytes = 96u << 10;  // cluster kernels: shared-memory stage per CTA
constexpr int kClusterMaxRanks = 16;              // cluster kernels: ranks per cluster (one CTA each)
constexpr int kClusterBatch = 8;                  // cluster kernels: input vectors a thread keeps in flight

// Host-side launch entry points (kernels.cu).
cudaError_t launch_allreduce(const Params& p, rra_dtype_t dtype, int kind, int threads, cudaStream_t stream,
                             bool cooperative = true, bool pdl = false);
cudaError_t occupancy(rra_dtype_t dtype, int kind, int threads, int* blocks_per_sm);
// One-shot / two-shot through distributed shared memory (cluster.cu): one
// cluster of N CTAs per slice of p.per_cta vectors (a multiple of N for the
// two-shot).  kClusterOneshot / kClusterTwoshot: p.ctas_per_rank slices, one
// cluster each.  kClusterTwoshotPipe: p.ctas_per_rank persistent clusters
// over p.nsteps slices of at most threads * kClusterBatch vectors.
// kClusterOneshotMulti / kClusterTwoshotMulti: N > 16, clusters of 16 CTAs,
// CTA j hosting ranks j, j + 16, ...; the two-shot's slice is a multiple of 16.
// The ...MultiRes modes are the same kernels with the residual add of
// rra_allreduce_residual in their epilogue (launch_cluster_residual only).
// kClusterOneshotTma / kClusterTwoshotTma: kClusterOneshot / kClusterTwoshot
// with the push made by bulk copies (RRA_ATTR_CLUSTER_TMA); the ...MultiTma
// modes the same for more than 16 ranks.  kClusterOneshotTmaRes:
// kClusterOneshotTma with the residual add of rra_allreduce_residual in its
// epilogue (launch_cluster_tma_residual only).
enum { kClusterOneshot = 0, kClusterTwoshot = 1, kClusterTwoshotPipe = 2, kClusterOneshotMulti = 3,
       kClusterTwoshotMulti = 4, kClusterOneshotMultiRes = 5, kClusterTwoshotMultiRes = 6,
       kClusterOneshotTma = 7, kClusterTwoshotTma = 8, kClusterOneshotMultiTma = 9, kClusterTwoshotMultiTma = 10,
       kClusterOneshotTmaRes = 11 };
size_t cluster_stage_bytes(const Params& p, int mode);
cudaError_t launch_cluster(const Params& p, rra_dtype_t dtype, int mode, int threads, cudaStream_t stream, bool pdl);
int cluster_max_active(rra_dtype_t dtype, int mode, int nranks, int threads, size_t smem);
// ReduceScatter, AllGather, Broadcast, Reduce through distributed shared
// memory (coll.cu): one cluster of N CTAs per slice of p.per_cta vectors of
// a block of p.count elements (p.nvec vectors), p.ctas_per_rank slices.
enum {
    kCollReduceScatter = 0,
    kCollAllGather = 1,
    kCollBroadcast = 2,
    kCollReduce = 3,
    kCollBroadcastSplit = 4,  // two hops: scatter from the root, then every CTA pushes its part
    kCollReduceSplit = 5      // two hops: ReduceScatter, then every owner pushes to the root
};
size_t coll_stage_bytes(const Params& p, int op);
// bulk: ReduceScatter / AllGather / Broadcast up to 16 ranks on the
// bulk-copy kernels (the caller has checked that every input they read is
// device memory of this GPU, and for ReduceScatter that a block is whole
// 16-byte vectors); otherwise the st.async kernels.  store_bulk (with bulk): the outputs are
// written by bulk copies as well (the caller has checked that every output
// is device memory of this GPU and that a block is whole 16-byte vectors).
bool coll_has_bulk(int op, int nranks);
const char* coll_kernel_name(int op, int nranks, bool bulk, bool store_bulk);
cudaError_t launch_coll(const Params& p, rra_dtype_t dtype, int op, int threads, cudaStream_t stream, bool pdl,
                        bool bulk, bool store_bulk);
int coll_max_active(rra_dtype_t dtype, int op, int nranks, int threads, size_t smem, bool bulk);
// AllReduce + residual add on the public device API (fused.cu): the cluster
// AllReduce's launch shape; cluster c handles slices c, c + G, ... of
// p.nsteps slices (G = p.ctas_per_rank), one epoch each.
struct FusedParams {
    Params base;
    const void* resid[kMaxRanks];  // rank r's residual stream (count elements)
};
size_t residual_stage_bytes(const Params& p, bool two_shot);
// bulk: the pushes are the device API's bulk sends (TMA copies).
cudaError_t launch_residual(const FusedParams& f, rra_dtype_t dtype, bool two_shot, bool bulk, int threads,
                            cudaStream_t stream, bool pdl);
int residual_max_active(rra_dtype_t dtype, bool two_shot, bool bulk, int nranks, int threads, size_t smem);
// The same above 16 ranks (cluster.cu): f.base planned as for the many-rank
// cluster AllReduce (kClusterOneshotMulti / kClusterTwoshotMulti).
cudaError_t launch_cluster_residual(const FusedParams& f, rra_dtype_t dtype, bool two_shot, int threads,
                                    cudaStream_t stream, bool pdl);
// The one-shot of up to 16 ranks on bulk copies with the residual add in its
// epilogue (cluster.cu): f.base planned as for the cluster AllReduce's
// kClusterOneshotTma.
cudaError_t launch_cluster_tma_residual(const FusedParams& f, rra_dtype_t dtype, int threads, cudaStream_t stream,
                                        bool pdl);
cudaError_t launch_init(char* base, size_t total, const rra_layout_t& lay, int nranks,
                        cudaStream_t stream);

}  // namespace rra
