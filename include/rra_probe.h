/*
 * rra_probe.h -- single-GPU latency-floor probes (C ABI).
 *
 * "Every Microsecond Matters", Sec. VI, models the speed-of-light latency of
 * a small push AllReduce as L_SoL = 2 * L_L2_RTT + L_remote_store: one L2
 * round trip to load the input, one store into the peer's scratch, one L2
 * round trip to read it back (the output store is not waited on).  On one GPU
 * the "remote" store is a store from one SM that another SM observes through
 * L2.  These probes measure both terms on the GPU they run on:
 *
 *  - L_L2_RTT by a dependent pointer chase through an L2-resident buffer that
 *    is larger than L1 (not by a memory fence, whose latency includes draining
 *    the memory pipeline);
 *  - L_store->poll as half the round trip of a fence-free ping-pong between
 *    two CTAs that sit on different SMs.
 *
 * All waits are bounded by a time limit; a probe that gives up returns
 * RRA_ERR_TIMEOUT instead of hanging.
 */
#ifndef RRA_PROBE_H
#define RRA_PROBE_H

#include "rra.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Dependent-load chase over a random cycle of 8-byte words in a device
 * buffer of `buf_bytes` (allocated and freed here; >= 64 KiB).  One warm pass
 * brings the buffer into L2, then one thread follows `hops` pointers with
 * L1-bypassing loads.  Output: mean ns per hop.  `seed` picks the cycle.
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_OOM, RRA_ERR_CUDA. */
rra_status_t rra_probe_l2_chase(size_t buf_bytes, uint64_t hops, uint64_t seed,
                                double* ns_per_hop);

/* Fence-free ping-pong between CTA `cta_a` and CTA `cta_b` of a grid that
 * holds one CTA per SM (cooperative launch, so both are resident).  CTA a
 * stores i to a flag; CTA b polls until it sees i and stores i to a second
 * flag; CTA a polls that.  Output: mean ns per round trip over `iters`
 * exchanges after `iters`/8 warm-up exchanges, and the SM ids the two CTAs ran
 * on (they differ: one CTA per SM).  Errors: RRA_ERR_INVALID_ARG,
 * RRA_ERR_TIMEOUT (a wait passed 1 s), RRA_ERR_CUDA. */
rra_status_t rra_probe_pingpong(int cta_a, int cta_b, int iters,
                                double* ns_round_trip, int* sm_a, int* sm_b);

/* The same floor for the cluster kernels, whose ranks exchange data through
 * distributed shared memory.  Two CTAs of one thread-block cluster play
 * ping-pong with TMA bulk copies: each turn copies 128 bytes from an
 * L2-resident device buffer into the other CTA's shared memory, and the
 * copy's arrival completes that CTA's mbarrier, on which it waits.  Outputs:
 * mean ns per round trip over `iters` turns after `iters`/8 warm-up turns;
 * mean ns per cluster barrier (relaxed arrive, acquire wait) over `iters`
 * back-to-back barriers; the two SM ids.  Half the round trip (the input
 * read and the push in one) plus one cluster barrier (the one such a kernel
 * passes before its first push) is the floor of one push through shared
 * memory.  Errors: RRA_ERR_INVALID_ARG, RRA_ERR_OOM, RRA_ERR_TIMEOUT (a wait
 * passed 1 s), RRA_ERR_CUDA. */
rra_status_t rra_probe_dsmem_pingpong(int iters, double* ns_round_trip, double* ns_cluster_barrier,
                                      int* sm_a, int* sm_b);

/* Launch one empty kernel (1 CTA, 32 threads) on `stream`, to measure launch
 * and graph-node overhead next to the AllReduce. */
rra_status_t rra_probe_empty_kernel(rra_stream_t stream);

/* Launch `ctas` x `threads` empty CTAs on `stream` (cooperative if
 * `cooperative`), with a 1152-byte parameter block if `big_params` (the size
 * of the AllReduce kernels' parameters) or none: separates launch and
 * graph-node cost by grid shape, parameter size and launch kind. */
rra_status_t rra_probe_launch_shape(int ctas, int threads, int big_params, int cooperative, rra_stream_t stream);

/* Launch one empty kernel of `ctas` x `threads` on `stream` as the AllReduce
 * kernels launch: in clusters of `cluster` CTAs (1: no cluster; up to 8,
 * dividing `ctas`) and, if `pdl`, with programmatic dependent launch; the
 * kernel releases its successor and waits for its predecessor as the
 * AllReduce kernels do (griddepcontrol; a one-cluster grid releases at
 * entry, a larger one after its wait), nothing else.  A chain of these in a CUDA graph gives
 * the per-call floor of back-to-back dependent calls of that shape.
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_CUDA. */
rra_status_t rra_probe_launch_chain(int ctas, int threads, int cluster, int pdl, rra_stream_t stream);

/* Number of SMs of the current device. */
rra_status_t rra_probe_sm_count(int* sms);

/* The host link that the host-buffer AllReduce (rra_allreduce_host,
 * rra_allreduce_mapped, zero copy) runs over: two pinned, device-mapped host
 * buffers of `bytes` each (allocated and freed here; 64 KiB to 1 GiB, a
 * multiple of 16) streamed with 16-byte loads and stores.  Outputs, in GB/s
 * of `bytes` per launch (mean over `iters` launches after two warm-ups):
 * read_gbps, the device reading the first buffer; write_gbps, the device
 * writing the second; copy_gbps, the device copying the first into the
 * second, one vector in flight per thread, so that reads and writes overlap
 * (bytes per second in each direction).  The copy reaches its steady rate
 * from about 16 MiB; smaller buffers spend a larger share filling and
 * draining.  The copy is checked on the host afterwards.
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_OOM, RRA_ERR_CUDA (a launch failed or
 * the copied buffer differs). */
rra_status_t rra_probe_host_link(size_t bytes, int iters, double* read_gbps, double* write_gbps,
                                 double* copy_gbps);

#ifdef __cplusplus
}
#endif

#endif /* RRA_PROBE_H */
