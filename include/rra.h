/*
 * rra.h -- barrier-free AllReduce over N virtual ranks on one GPU (C ABI).
 *
 * The operation is the AllReduce of "Every Microsecond Matters: Achieving
 * Near Speed-of-Light Latency in GPU Collectives" (arXiv 2607.16100),
 * Sec. III-A: every rank r contributes a vector send[r] of `count` elements
 * and receives, in recv[r], the element-wise sum over all ranks.  The four
 * algorithms are the paper's barrier-free designs (Sec. IV): one-shot push
 * with the LL protocol, one-shot push with sentinel-initialised scratch,
 * two-shot (ReduceScatter + AllGather) with bidirectional double buffering,
 * and the two-shot LL128-atomic variant (Fig. 5).  No global barrier is used:
 * every wait is on the arrival of data.
 *
 * Virtual ranks.  The N ranks live on ONE GPU.  Rank r is a group of CTAs
 * that owns window r of one symmetric device allocation (window r starts
 * `stride` bytes after window r-1), the single-GPU analogue of the symmetric
 * memory windows of Sec. II-B.  A rank reads only its own input and its own
 * window and writes only peers' windows and its own output; L2 is the point
 * of coherence between ranks.  All CTAs of a call are launched cooperatively
 * so that every polling CTA is co-resident with the CTAs it waits for.
 *
 * Results.  recv[r][i] = send[0][i] + send[1][i] + ... + send[N-1][i], the
 * same value for every r.  One-shot and two-shot add in rank order 0..N-1
 * with a binary32 running value for RRA_FP32/RRA_BF16 (bfloat16 results are
 * rounded to nearest-even once at the end) and binary64 for RRA_FP64; they
 * are bit-for-bit deterministic.  RRA_LL128_ATOMIC adds with hardware
 * atomics in an unspecified order into binary32 (binary64 for RRA_FP64)
 * accumulators; every rank still receives the identical bit pattern.
 *
 * Streams and graphs.  A call only enqueues work on `stream` (no host
 * synchronisation, no host-to-device copies), so it can be captured into a
 * CUDA graph; the per-call epoch lives in device memory and advances on every
 * replay.  Calls on one communicator must be ordered on one stream.
 *
 * Errors.  Every function returns an rra_status_t.  Argument and CUDA launch
 * errors are returned directly.  Errors found on the device (a poll that ran
 * past its time limit) are recorded in a device status word: they do not
 * fault the GPU, later calls on the same communicator become no-ops on the
 * device, rra_comm_status() reports them, and the communicator stays
 * poisoned (RRA_ERR_POISONED) until rra_comm_reset().
 *
 * Bulk-copy pushes stay on one GPU.  Some cluster kernels push by TMA bulk
 * copies with cluster multicast (cp.async.bulk ... .multicast::cluster) that
 * read straight from the callers' input buffers: the cluster one-/two-shot
 * AllReduce and the four collectives at every rank count, and the fused
 * residual AllReduce up to 16 ranks; AllGather and Broadcast also write
 * their outputs by bulk copies (then every output must be device memory of
 * the current GPU too).  A call uses them only when (a) every
 * buffer such a copy reads is device memory of the current GPU -- checked with
 * cudaPointerGetAttributes at both ends of the range read, the result of a
 * passing check remembered for the last 8 sets of input pointers of the
 * communicator -- and (b) the process holds no active context on any other
 * GPU.  Host buffers (rra_allreduce_host, rra_allreduce_mapped), another
 * GPU's memory, managed memory, and processes that also drive other GPUs
 * always get the st.async push (the same results).  rra_comm_last_kernel
 * names the kernel a call launched.
 */
#ifndef RRA_H
#define RRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                     /* same type as cudaStream_t */
typedef struct CUstream_st* rra_stream_t;

typedef struct rra_comm* rra_comm_t;    /* opaque communicator */

#define RRA_MAX_RANKS 64

typedef enum {
    RRA_OK = 0,
    RRA_ERR_INVALID_ARG = 1,     /* bad pointer, size, dtype, algo, alignment */
    RRA_ERR_CUDA = 2,            /* a CUDA runtime call failed */
    RRA_ERR_OOM = 3,             /* device allocation failed */
    RRA_ERR_NOT_CORESIDENT = 4,  /* N ranks cannot all be resident at once */
    RRA_ERR_TIMEOUT = 5,         /* a device-side poll gave up (see status) */
    RRA_ERR_POISONED = 6         /* an earlier device error; call rra_comm_reset */
} rra_status_t;

typedef enum { RRA_FP32 = 0, RRA_BF16 = 1, RRA_FP64 = 2 } rra_dtype_t;

typedef enum {
    RRA_ONESHOT_LL = 0,        /* Sec. IV "LL": data and epoch flag share one atomic word */
    RRA_ONESHOT_SENTINEL = 1,  /* Sec. IV "Sentinel": scratch pre-filled with -NaN, polled */
    RRA_TWOSHOT_DBUF = 2,      /* Sec. III-A two-shot + Sec. IV double buffering, Fig. 4 */
    RRA_LL128_ATOMIC = 3,      /* Fig. 5: atomic adds into the owner's lines, counter == N-1 */
    RRA_ONESHOT_BARRIER = 4,   /* BASELINE, not barrier-free: plain stores + two flag barriers
                                  per step (Sec. III-B, the design the paper replaces) */
    RRA_TWOSHOT_DIRECT = 5,    /* two-shot whose AllGather stores the reduced partition
                                  straight into every rank's output (outputs treated as
                                  registered symmetric buffers, Sec. II-B): RS as
                                  RRA_TWOSHOT_DBUF, no AG scratch, one hop per step */
    RRA_AUTO = 6,              /* pick by rank count and message size (rra_select_algo);
                                  may pick a sentinel algorithm when clusters cannot be
                                  scheduled, so inputs must not hold the all-ones
                                  pattern */
    RRA_ONESHOT_CLUSTER = 7,   /* one-shot push through distributed shared memory: one
                                  thread-block cluster of N CTAs per slice (CTA r = rank r);
                                  the push -- a TMA bulk copy of the slice with cluster
                                  multicast (default, RRA_ATTR_CLUSTER_TMA, only on inputs
                                  in this GPU's device memory: see "Bulk-copy pushes" above),
                                  or st.async stores -- completes the peers' mbarrier (arrival of the
                                  bytes is the signal); no state between calls.  For N > 16 the clusters have 16 CTAs and
                                  CTA j hosts ranks j, j+16, ... (pushes go to the 15 other
                                  CTAs; still the rank-order sum of all N) */
    RRA_TWOSHOT_CLUSTER = 8,   /* two-shot through distributed shared memory: rank r pushes
                                  partition q of its slice to CTA q only (ReduceScatter),
                                  CTA q adds the N contributions in rank order and stores
                                  the result into every rank's output (AllGather as direct
                                  stores, as RRA_TWOSHOT_DIRECT); HBM carries only the
                                  inputs read once and the outputs written once.  N > 16:
                                  16-CTA clusters, CTA q reduces part q over all N ranks */
    RRA_TWOSHOT_BARRIER = 9    /* BASELINE, not barrier-free: two-shot with plain stores and
                                  two flag barriers per step (ReduceScatter, barrier, reduce
                                  + AllGather stores, barrier, gather; Sec. III-B's design
                                  applied to Sec. III-A's two-shot); rank-order sums */
} rra_algo_t;

/* Communicator attributes (rra_comm_set_attr / rra_comm_get_attr). */
typedef enum {
    RRA_ATTR_CTAS_PER_RANK = 0,    /* 0 = chosen per call from the message size; for the
                                      persistent cluster two-shot, a cap on its clusters */
    RRA_ATTR_POLL_TIMEOUT_MS = 1,  /* limit of every device-side wait (default 1000) */
    RRA_ATTR_THREADS = 2,          /* largest threads per CTA: 64, 128 (default) or 256; while
                                      it is not set, the cluster two-shot may use 256 for
                                      messages up to ~1-2 MiB per rank.  RRA_TWOSHOT_DBUF and
                                      RRA_TWOSHOT_DIRECT use at most 128 (their kernels are
                                      built for 4 CTAs of 128 threads per SM) */
    RRA_ATTR_TWOSHOT_CHUNK = 3,    /* bytes per rank per two-shot step (RRA_TWOSHOT_DBUF,
                                      RRA_TWOSHOT_DIRECT); 0 (default) = one 16-byte position
                                      per thread of the largest co-resident grid, at most the
                                      step whose live ReduceScatter scratch over all windows
                                      is ~32 MiB, within the per-window scratch cap */
    RRA_ATTR_LL128_CHUNK = 4,      /* bytes per rank per LL128-atomic step; 0 = the step
                                      whose live scratch over all windows is ~64 MiB (stays
                                      in L2), within the per-window scratch cap */
    RRA_ATTR_ONESHOT_CHUNK = 5,    /* bytes per rank per one-shot step, 0 = largest */
    RRA_ATTR_ONESHOT_WIDE = 6,     /* the one-shot's polls and the LL128-atomic kernel's adds
                                      and polls split a position's sources over threads:
                                      -1 auto (N >= 16, default), 0 off, 1 on */
    RRA_ATTR_COOPERATIVE = 7,      /* 1 (default): cooperative launch, so the driver
                                      guarantees that all CTAs are resident together;
                                      0: plain launch of the same occupancy-checked grid
                                      (progress then relies on no other work holding the
                                      SMs for longer than the poll time limit).  Either
                                      way, a global-memory one-shot with one CTA per rank
                                      on 2-16 CTAs launches as one thread-block cluster,
                                      which keeps its ranks on one GPC and is resident
                                      together by construction */
    RRA_ATTR_PDL = 8,              /* 1 (default): programmatic dependent launch, so
                                      the next kernel on the stream is scheduled while
                                      this one drains; each kernel waits
                                      (griddepcontrol.wait) for its predecessor before
                                      touching memory.  0: plain stream order */
    RRA_ATTR_CLUSTER_SLICE = 9,    /* cluster kernels: bytes per rank per slice (one cluster
                                      per slice), a multiple of 16, at most 98304; clamped to
                                      the 96 KiB shared-memory stage (N x slice for the
                                      one-shot, slice for the two-shot, rounded up to N
                                      vectors).  0 (default): one 16-byte vector per thread
                                      for small messages, else about two CTAs per SM, at
                                      most 8 vectors per thread */
    RRA_ATTR_CLUSTER_PIPE = 10,    /* cluster two-shot on the persistent, double-buffered
                                      kernel (as many clusters as fit at once, each looping
                                      over slices; a receiver's arrival on the sender's
                                      "empty" mbarrier is the credit for the next push):
                                      0 (default) never, -1 when the slices do not fit in
                                      one wave, 1 whenever the slice allows (at most 8
                                      vectors per thread and a 2 x slice stage <= 96 KiB).
                                      Off by default: on GB300 it was up to 2.3x slower
                                      than one cluster per slice at 4-64 MiB per rank */
    RRA_ATTR_HOST_ZERO_COPY = 11,  /* rra_allreduce_host: 1 (default) when every buffer is
                                      pinned host memory the device can address, the
                                      kernel reads and writes it in place (no staging);
                                      0: always stage through device buffers */
    RRA_ATTR_COLL_SPLIT = 12,      /* rra_broadcast / rra_reduce in two hops (the root
                                      scatters its slice and every CTA forwards its part /
                                      ReduceScatter, then every owner sends to the root):
                                      -1 (default) when nranks >= 3 and the message is at
                                      least 256 KiB, except a Broadcast that runs on bulk
                                      copies both ways and a Reduce on bulk copies (see
                                      "The other collectives"), which stay one call of their
                                      own shape; 0 never, 1 always; up to 16 ranks */
    RRA_ATTR_CLUSTER_TMA = 13      /* cluster one-/two-shot AllReduce with the push made
                                      by the TMA engine: bulk copies from a rank's input
                                      into the peers' shared memory (multicast to all CTAs
                                      for the one-shot, one copy per partition owner for
                                      the two-shot; above 16 ranks one per hosted rank);
                                      also the fused residual AllReduce (up to 16 ranks)
                                      and the four collectives.  -1 (default) and 1: on
                                      (faster at every N and size measured but the
                                      smallest two-shot calls) for calls whose inputs pass
                                      the check of "Bulk-copy pushes" above; 0: st.async
                                      pushes always */
} rra_attr_t;

/* Scratch layout of one window (bytes), as planned for (nranks, max_bytes).
 * The per-algorithm caps default to the paper's scratch sizes (Sec. VII,
 * Fig. 12): 4 MiB for one-shot, 64 MiB for two-shot and LL128-atomic. */
typedef struct {
    int nranks;
    size_t max_bytes;
    size_t ll_chunk;        /* one-shot LL payload bytes per rank per step */
    size_t ll_bytes;        /* LL region: 2 parities x N slots x 2*ll_chunk */
    size_t os_chunk;        /* one-shot sentinel payload bytes per rank per step */
    size_t os_bytes;        /* sentinel region: 2 x N x os_chunk */
    size_t ts_part;         /* two-shot partition bytes per owner per step */
    size_t ts_bytes;        /* RS + AG regions: 2 x (2 x N x ts_part) */
    size_t la_part;         /* LL128-atomic partition payload bytes per owner per step */
    size_t la_bytes;        /* accumulators + counters + LL-encoded AllGather slots */
    size_t window_stride;   /* bytes between consecutive windows */
    size_t ctrl_bytes;      /* control block before window 0 */
    size_t total_bytes;     /* ctrl_bytes + nranks * window_stride */
    size_t bf_bytes;        /* barrier baseline flags: 64 CTAs x 64 ranks x 4 B */
    size_t bd_chunk;        /* barrier baseline payload bytes per rank per step */
    size_t bd_bytes;        /* barrier baselines' data: 2 x N x bd_chunk (one-shot cap);
                               the two-shot baseline's AllGather slots are the second half */
} rra_layout_t;

/*
 * rra_comm_create: allocate the symmetric windows and initialise them.
 *   nranks     number of virtual ranks, 2 <= nranks <= RRA_MAX_RANKS.
 *   max_bytes  largest message (count * element size) a call may pass, > 0.
 *   out        receives the communicator; unchanged on error.
 * Uses the current CUDA device.  Allocates once (cudaMalloc of
 * layout.total_bytes, and one pinned, device-mapped host word into which
 * device code mirrors the first error, so that rra_allreduce_host can read
 * it without a copy); fills sentinel regions with all-one bytes, LL flags,
 * accumulators and counters with zero, sets the epoch to 1 and synchronises.
 * Environment overrides read here: RRA_POLL_TIMEOUT_MS, RRA_CTAS_PER_RANK,
 * RRA_THREADS, RRA_SCRATCH_ONESHOT, RRA_SCRATCH_TWOSHOT (bytes).
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_OOM, RRA_ERR_CUDA,
 * RRA_ERR_NOT_CORESIDENT (fewer than nranks CTAs fit on the GPU at once).
 */
rra_status_t rra_comm_create(int nranks, size_t max_bytes, rra_comm_t* out);

/*
 * rra_allreduce: enqueue one AllReduce-sum on `stream` (Sec. III-A).
 *   send[r]  device pointer to rank r's `count` input elements (r < nranks).
 *   recv[r]  device pointer to rank r's `count` output elements.
 *            send and recv are host arrays of nranks device pointers; they are
 *            copied into the kernel's parameters, so they may be freed on
 *            return.  Every pointer must be 16-byte aligned.  recv[r] may equal
 *            send[r] (in place); buffers of different ranks must not overlap.
 *   count    elements per rank; count == 0 returns RRA_OK without a launch;
 *            count * element size must not exceed max_bytes.
 *   dtype    element type; algo: one of rra_algo_t.
 *   stream   CUDA stream (NULL = legacy default stream).
 * The caller owns all buffers and must keep them alive until the work on
 * `stream` completes.  RRA_ONESHOT_SENTINEL and RRA_TWOSHOT_DBUF require
 * that no input element has the all-ones bit pattern (the sentinel, a
 * negative NaN, Sec. IV "Sentinel"); such an input makes the call time out.
 * The cluster algorithms return RRA_ERR_NOT_CORESIDENT if the device cannot
 * schedule a cluster of min(nranks, 16) CTAs with a 96 KiB stage each.
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_POISONED, RRA_ERR_CUDA,
 * RRA_ERR_NOT_CORESIDENT.
 */
rra_status_t rra_allreduce(rra_comm_t comm, const void* const send[], void* const recv[],
                           size_t count, rra_dtype_t dtype, rra_algo_t algo,
                           rra_stream_t stream);

/*
 * rra_allreduce_host: the same operation on HOST buffers, end to end.
 * send[r]/recv[r] are host pointers, 16-byte aligned.  If every one of them
 * is pinned host memory that the device can address (cudaHostAlloc'd or
 * registered; on GB300 the GPU reaches it over the coherent NVLink-C2C link
 * to the Grace CPU) and RRA_ATTR_HOST_ZERO_COPY is 1 (default), the kernel
 * reads the inputs and writes the outputs in host memory directly; such a
 * call moves nranks * count elements each way over the host link, whose
 * rates rra_probe_host_link (rra_probe.h) measures, and the cluster two-shot
 * then takes 4 KiB slices, which keep more of that link busy.
 * Otherwise the call copies every send[r] to device staging buffers owned
 * by the communicator (allocated on first use: 2 * nranks * max_bytes), runs
 * rra_allreduce, and copies every recv[r] back (one cudaMemcpyAsync per rank
 * and direction).  Either way it synchronises `stream` before returning.
 * Errors: as rra_allreduce, plus RRA_ERR_OOM for the staging buffers, plus
 * any device-side error of this call (the status word is read after the
 * synchronisation).
 */
rra_status_t rra_allreduce_host(rra_comm_t comm, const void* const send[], void* const recv[],
                                size_t count, rra_dtype_t dtype, rra_algo_t algo,
                                rra_stream_t stream);

/*
 * Resolve host buffers once for repeated end-to-end calls (the analogue of
 * registering buffers with a communicator, Sec. II-B): dev[i] receives the
 * device address of host[i] when host[i] points into pinned host memory
 * that the device can address, else NULL (also for a NULL host[i]).
 * 0 <= n <= 2 * RRA_MAX_RANKS.  No communicator is involved and nothing is
 * allocated; the addresses stay valid while the host memory stays pinned.
 */
rra_status_t rra_host_device_ptrs(int n, const void* const host[], void* dev[]);

/*
 * rra_allreduce_host on buffers resolved by rra_host_device_ptrs (every
 * send[r] and recv[r] a device address of pinned host memory): runs
 * rra_allreduce on them, so the kernel reads and writes host memory
 * directly, then synchronises `stream` and returns the device status of the
 * communicator (RRA_OK, or the first device-side error, which poisons it).
 * Arguments and errors otherwise as rra_allreduce.
 */
rra_status_t rra_allreduce_mapped(rra_comm_t comm, const void* const send[], void* const recv[],
                                  size_t count, rra_dtype_t dtype, rra_algo_t algo,
                                  rra_stream_t stream);

/*
 * The other collectives.  The paper text (Sec. III-A, opening) notes that
 * AllReduce is commonly built from ReduceScatter + AllGather or from
 * Reduce + Broadcast; its review (summary) adds that the same barrier-free
 * primitives serve these four.  Here all four run one thread-block cluster
 * of nranks CTAs per slice, CTA r acting for rank r, and exchange data
 * through distributed shared memory: a push is an st.async into a peer's
 * shared memory that completes the peer's mbarrier, and the only wait is a
 * bounded wait on one's own mbarrier (data arrival is the signal).  Up to 16
 * ranks, when every input a call reads is device memory of this GPU, the
 * pushes are TMA bulk copies straight from the inputs instead: AllGather and
 * Broadcast one copy of the slice with cluster multicast into every CTA;
 * ReduceScatter one copy per owner (only when count x element size is a
 * multiple of 16, so that every block starts 16-byte aligned); Reduce one
 * copy per partition owner, each owner then storing its rank-order sums of
 * its partition into the root's output.  AllGather (blocks of 4 KiB and up)
 * and Broadcast (256 KiB and up) on bulk copies also write their outputs
 * from shared memory by bulk copies (one per block, issued by one thread)
 * when every output is device memory of this GPU and count x element size
 * is a multiple of 16, so that no copy writes past its block; otherwise
 * every thread stores vectors.  Above
 * 16 ranks (the cluster limit) a cluster has 16 CTAs and CTA j acts for
 * ranks j, j + 16, j + 32, ...; pushes between ranks of one CTA are plain
 * shared-memory stores.  Nothing persists between calls.
 *
 * Common rules: any nranks of the communicator (2..64).  Broadcast and
 * Reduce take two hops for large messages up to 16 ranks
 * (RRA_ATTR_COLL_SPLIT), one hop above.  send/recv are host arrays of
 * nranks device pointers, each 16-byte
 * aligned where it is used.  count == 0 returns RRA_OK without a launch.
 * Sums add the ranks in order 0..nranks-1 with a binary32 running value for
 * binary32 and bfloat16 (rounded to nearest-even once) and binary64 for
 * binary64, exactly like the fixed-order AllReduce kernels.  Errors: as
 * rra_allreduce (RRA_ERR_NOT_CORESIDENT if the device cannot schedule a
 * cluster of min(nranks, 16) CTAs with a 96 KiB stage each).
 *
 * rra_reduce_scatter: send[r] holds nranks * count elements (block q =
 *   elements [q * count, (q + 1) * count)); recv[r] receives count elements,
 *   the sum over ranks of block r.  nranks * count * element size must not
 *   exceed max_bytes.  recv[r] may be send[r] + r * count (in place, when
 *   that address is 16-byte aligned); buffers must not overlap otherwise.
 */
rra_status_t rra_reduce_scatter(rra_comm_t comm, const void* const send[], void* const recv[],
                                size_t count, rra_dtype_t dtype, rra_stream_t stream);

/* rra_all_gather: send[r] holds count elements; recv[r] receives
 * nranks * count elements, block p being a copy of send[p].
 * nranks * count * element size must not exceed max_bytes.  send[r] may be
 * recv[r] + r * count (in place, when 16-byte aligned). */
rra_status_t rra_all_gather(rra_comm_t comm, const void* const send[], void* const recv[],
                            size_t count, rra_dtype_t dtype, rra_stream_t stream);

/* rra_broadcast: every recv[r] (count elements) receives a copy of
 * send[root].  Only send[root] is read; the other send entries may be NULL.
 * recv[root] may equal send[root].  0 <= root < nranks. */
rra_status_t rra_broadcast(rra_comm_t comm, int root, const void* const send[], void* const recv[],
                           size_t count, rra_dtype_t dtype, rra_stream_t stream);

/* rra_reduce: recv[root] receives the sum over ranks of send[r] (count
 * elements each).  Only recv[root] is written; the other recv entries may
 * be NULL.  recv[root] may equal send[root].  0 <= root < nranks. */
rra_status_t rra_reduce(rra_comm_t comm, int root, const void* const send[], void* const recv[],
                        size_t count, rra_dtype_t dtype, rra_stream_t stream);

/*
 * rra_allreduce_residual: AllReduce with the residual add of a
 * tensor-parallel layer fused into it.
 *     recv[r][i] = round( (send[0][i] + ... + send[N-1][i]) + residual[r][i] )
 * The ranks are added in order 0..N-1 with a binary32 running value for
 * binary32 and bfloat16 (binary64 for binary64), the residual is added to
 * the running value, and bfloat16 is rounded once, at the end.  The paper
 * (Abstract; Sec. I, contributions; Fig. 6-9) builds a device-side API for
 * custom collective kernels; this kernel is written on this library's
 * restatement of it, include/rra_device.cuh.
 *   send, residual, recv: host arrays of nranks device pointers, 16-byte
 *   aligned, count elements each; recv[r] may equal send[r] or residual[r].
 * Shape: one thread-block cluster of nranks CTAs per slice; each rank
 * pushes its slice to every peer's shared memory (one-shot) or each
 * partition to its owner (two-shot), the owner then writing every rank's
 * output with that rank's residual (outputs and residuals are then treated
 * as registered symmetric buffers, as by RRA_TWOSHOT_DIRECT).  The shape is
 * the one RRA_AUTO's cluster AllReduce takes (rra_select_algo); the pushes
 * are the device API's bulk sends unless RRA_ATTR_CLUSTER_TMA is 0.  Up to
 * 16 ranks, at one-shot sizes with the bulk-copy push and one slice per
 * cluster (RRA_ATTR_CTAS_PER_RANK unset), the kernel is the cluster
 * AllReduce's own bulk-copy one-shot with the residual add in its epilogue
 * ("cluster_tma_kernel<one-shot, residual>"), not the device-API kernel.
 * Above 16 ranks: the
 * many-rank cluster AllReduce (16-CTA clusters, CTA j acting for ranks j,
 * j + 16, ...; one-shot while 16 * nranks * count * element size <= 1 MiB)
 * with the residual add in its epilogue instead of the device-API kernel.
 * RRA_ATTR_CLUSTER_SLICE and RRA_ATTR_THREADS apply; up to 16 ranks
 * RRA_ATTR_CTAS_PER_RANK, when set, caps the clusters, each then looping
 * over several slices.  Errors: as rra_allreduce.
 */
rra_status_t rra_allreduce_residual(rra_comm_t comm, const void* const send[], const void* const residual[],
                                    void* const recv[], size_t count, rra_dtype_t dtype,
                                    rra_stream_t stream);

/* Synchronise the device and return the device status word: RRA_OK, or the
 * first device-side error (e.g. RRA_ERR_TIMEOUT); RRA_ERR_POISONED if an
 * earlier call of this function saw one and no rra_comm_reset followed.  A
 * device error poisons the communicator until rra_comm_reset(). */
rra_status_t rra_comm_status(rra_comm_t comm);

/* Where the first device-side error was recorded: synchronises the device
 * and stores the virtual rank and the chunk step of the call that recorded it
 * (-1 and -1 when the status word is clear).  Returns RRA_OK (also when an
 * error is recorded: read it with rra_comm_status), RRA_ERR_INVALID_ARG for
 * NULL arguments, RRA_ERR_CUDA. */
rra_status_t rra_comm_error_site(rra_comm_t comm, int* rank, int* step);

/* The kernel (as rra_comm_plan_kernel names it, e.g.
 * "cluster_tma_kernel<one-shot>" or "coll_bulk_kernel<all_gather>") that the
 * last call enqueued on this communicator launched: AllReduce, host and
 * mapped AllReduce, the four collectives, the fused residual AllReduce.
 * "none" before the first call.  *name points to a static string. */
rra_status_t rra_comm_last_kernel(rra_comm_t comm, const char** name);

/* Synchronise the device, re-initialise every window (sentinels, flags,
 * accumulators, counters), the epoch and the status word, and clear the
 * poison and any injected fault. */
rra_status_t rra_comm_reset(rra_comm_t comm);

/* Synchronise the device and free everything the communicator owns. */
rra_status_t rra_comm_destroy(rra_comm_t comm);

/* Attributes: see rra_attr_t.  Invalid values return RRA_ERR_INVALID_ARG. */
rra_status_t rra_comm_set_attr(rra_comm_t comm, rra_attr_t attr, int64_t value);
rra_status_t rra_comm_get_attr(rra_comm_t comm, rra_attr_t attr, int64_t* value);

/* The window layout of an existing communicator. */
rra_status_t rra_comm_layout(rra_comm_t comm, rra_layout_t* out);

/* Plan a layout without a GPU (pure host arithmetic).  scratch_oneshot and
 * scratch_twoshot are the per-window caps in bytes (0 = the paper's 4 MiB /
 * 64 MiB).  Errors: RRA_ERR_INVALID_ARG. */
rra_status_t rra_plan_layout(int nranks, size_t max_bytes, size_t scratch_oneshot,
                             size_t scratch_twoshot, rra_layout_t* out);

/* The kernel (the __global__ function, and its variant) that rra_allreduce
 * launches for this call on this communicator when its buffers are device
 * memory of this GPU, e.g. "cluster_tma_kernel<one-shot>" -- the name a
 * profiler's launch list shows.
 * *name points to a static string.  Needs a device (plans the call,
 * including occupancy queries); count > 0. */
rra_status_t rra_comm_plan_kernel(rra_comm_t comm, size_t count, rra_dtype_t dtype, rra_algo_t algo,
                                  const char** name);

/* The algorithm RRA_AUTO uses for `nranks` ranks and `bytes` per rank (pure
 * host arithmetic).  The paper picks its kernel from measured crossovers in
 * message size and rank count (one-shot for small messages, two-shot once
 * they reach about a mebibyte at four ranks); these thresholds are the
 * crossovers measured on GB300 with CUDA-graph replay: with the bulk-copy
 * push (RRA_ATTR_CLUSTER_TMA) the cluster one-shot, up to 16 ranks, while
 * nranks^2 * bytes <= 8 MiB at nranks <= 2, 2 MiB at nranks <= 4, 4 MiB at
 * nranks <= 8 and 8 MiB above, and above 16 ranks while 16 * nranks * bytes
 * <= 16 MiB; with that attribute set to 0 on a communicator (for that
 * communicator's RRA_AUTO) while min(nranks, 16) * nranks * bytes <= 1 MiB;
 * the cluster two-shot above.
 * If the device cannot schedule the cluster shape, RRA_AUTO uses the choice
 * without cluster kernels: one-shot sentinel while nranks * bytes <= 1.5 MiB
 * (N <= 8); for N > 8 one-shot sentinel up to 4 KiB, LL128-atomic up to
 * 16 KiB (64 KiB at N = 64), the direct two-shot above. */
rra_status_t rra_select_algo(int nranks, size_t bytes, rra_dtype_t dtype, rra_algo_t* out);

/* Number of CTAs the next call of (count, dtype, algo) would launch, and the
 * number of chunk steps it would take; pure host arithmetic. */
rra_status_t rra_comm_plan_call(rra_comm_t comm, size_t count, rra_dtype_t dtype,
                                rra_algo_t algo, int* grid_ctas, int* steps);

/* Largest number of CTAs of (dtype, algo) that can be resident at once. */
rra_status_t rra_comm_max_coresident(rra_comm_t comm, rra_dtype_t dtype, rra_algo_t algo,
                                     int* ctas);

/* Optional in-kernel timing.  `dev_buf` is a device buffer of at least
 * 2 * (largest grid) uint64_t; while set, every CTA of every call writes its
 * %globaltimer start and end (ns) at dev_buf[2*cta] and dev_buf[2*cta+1].
 * NULL switches timing off.  The caller owns the buffer. */
rra_status_t rra_comm_set_timing(rra_comm_t comm, uint64_t* dev_buf);

/* Optional in-kernel trace (diagnostics).  `dev_buf` holds 6 uint64_t per
 * CTA of the largest grid; while set, thread 0 of every CTA records
 * %globaltimer at six points.  One-shot kernels (narrow variant): start,
 * control words read, first push issued, first position polled and reduced,
 * its output stored, end.  Cluster kernels (not the persistent two-shot):
 * start, first input in registers, first cluster barrier passed, pushes
 * issued, all contributions arrived, end.  Entries a kernel does not reach stay unchanged.  NULL switches
 * tracing off. */
rra_status_t rra_comm_set_trace(rra_comm_t comm, uint64_t* dev_buf);

/* Fault injection for tests (host-side injection only; no GPU fault): in every
 * call enqueued (or captured) while it is set, virtual rank `rank` skips every
 * store to its peers, so the peers' polls run into their time limit and record
 * RRA_ERR_TIMEOUT.  The rank travels in the kernel parameters.  rank = -1
 * clears it; rra_comm_reset also clears it.  Synchronises the device. */
rra_status_t rra_comm_inject_drop(rra_comm_t comm, int rank);

/* Barrier latency on this communicator's N ranks (Fig. 3 analogue, one
 * GPU): one CTA per rank runs `iters` flag barriers back to back (the barrier
 * of RRA_ONESHOT_BARRIER); output: mean ns per barrier between the first and
 * the last.  Synchronises the device.  Errors: RRA_ERR_INVALID_ARG (iters < 2),
 * RRA_ERR_POISONED, RRA_ERR_CUDA, and device errors as rra_comm_status. */
rra_status_t rra_comm_barrier_latency(rra_comm_t comm, int iters, double* ns_per_barrier);

/* Epoch of the next step (diagnostics and tests).  Each step of a call uses
 * one epoch; the LL flags carry its low 32 bits.  When a call's epochs would
 * reach a multiple of 2^31, the call first zeroes every LL flag region of every
 * window (the whole co-resident grid, followed by one bounded grid barrier)
 * and restarts at that multiple + 1, so no stale flag can match a live epoch.
 * rra_comm_set_epoch overwrites the epoch (epoch >= 1; it does not scrub, so
 * only move it forward to exercise that boundary).  Both synchronise the
 * device. */
rra_status_t rra_comm_get_epoch(rra_comm_t comm, uint64_t* epoch);
rra_status_t rra_comm_set_epoch(rra_comm_t comm, uint64_t epoch);

/* Text for a status code (static storage). */
const char* rra_status_string(rra_status_t status);

/* Library version, e.g. "0.1.0". */
const char* rra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RRA_H */
