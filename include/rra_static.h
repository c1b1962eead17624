/*
 * rra_static.h -- an AllReduce entry point that allocates nothing (C ABI).
 *
 * The paper has no counterpart to this entry point; it exists for callers of
 * this library that cannot allocate device memory when they need an
 * AllReduce: plug-ins and extensions whose host framework owns the GPU
 * allocator and forbids direct cudaMalloc/cudaFree (they are handed their
 * input and output buffers and nothing else), processes that reserve their
 * whole device-memory budget up front and may not grow it, and
 * latency-critical paths that must not pay for an allocation or for the
 * device-wide synchronisation that freeing memory can imply.
 */
#ifndef RRA_STATIC_H
#define RRA_STATIC_H

#include "rra.h"

#ifdef __cplusplus
extern "C" {
#endif

#define RRA_STATIC_MAX_RANKS 8              /* virtual ranks per call */
#define RRA_STATIC_MAX_BYTES (16u << 10)    /* count * element size per rank */

/*
 * rra_allreduce_static: the one-shot LL AllReduce-sum (same kernel and same
 * result as rra_allreduce with RRA_ONESHOT_LL: ranks added in order, bit for
 * bit), with no communicator and no allocation.  Its scratch is a file-scope
 * device array of about 4 MiB (a control block plus 8 windows of LL slots,
 * 512 KiB each) that every GPU loading this library holds until the process
 * exits.  The call issues no cudaMalloc, cudaFree or other allocating routine.
 *   nranks      2 <= nranks <= RRA_STATIC_MAX_RANKS.
 *   send, recv  host arrays of nranks device pointers (16-byte aligned), as for
 *               rra_allreduce; recv[r] may equal send[r].
 *   count       elements per rank; count * element size must not exceed
 *               RRA_STATIC_MAX_BYTES, otherwise RRA_ERR_INVALID_ARG and nothing
 *               is enqueued; count == 0 returns RRA_OK.
 *   dev_status  optional device pointer to one uint32_t: after the kernel, the
 *               call copies the device status into it on `stream` (0 = ok,
 *               RRA_ERR_TIMEOUT if a wait ran out).  NULL skips the copy.
 *   stream      CUDA stream.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and queries occupancy; make
 * that first call before any stream capture starts.  The array needs no
 * initialisation: all-zero, its state when the module loads, is the idle state.
 * Every call looks the address up again on the host, and redoes the set-up if
 * it moved (after cudaDeviceReset the module is loaded anew).
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  A call enqueues two kernels on `stream`: a one-CTA kernel
 * that, only if the previous call recorded an error, returns the whole array
 * to the idle state (so one failed call does not spoil the next), then the
 * AllReduce.  LL flags need no clearing after a successful call because every
 * call uses new epochs.  Calls whose work overlaps on the GPU (different
 * streams, or several host threads without ordering) race on the array and
 * give wrong results: order them on one stream.
 * Errors: RRA_ERR_INVALID_ARG, RRA_ERR_CUDA, RRA_ERR_NOT_CORESIDENT.
 */
rra_status_t rra_allreduce_static(int nranks, const void* const send[], void* const recv[], size_t count,
                                  rra_dtype_t dtype, uint32_t* dev_status, rra_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RRA_STATIC_H */
