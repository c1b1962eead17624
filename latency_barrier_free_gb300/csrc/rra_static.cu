// rra_static.cu -- an AllReduce entry point that allocates no device memory.
//
// Who needs it.  Some callers cannot call cudaMalloc at the moment they need
// an AllReduce, and cannot hold a communicator whose creation allocated for
// them either:
//  * plug-ins and extensions whose host framework owns the GPU allocator and
//    forbids direct cudaMalloc / cudaFree (all device memory must come from
//    the framework, and the plug-in is only handed input and output buffers);
//  * processes that reserve their whole device-memory budget up front and
//    may not grow it afterwards;
//  * latency-critical paths that must not pay for an allocation, or for the
//    device-wide synchronisation that freeing memory can imply.
// For them, rra_allreduce_static runs the one-shot LL AllReduce on scratch
// that is not allocated at all: it lives in the file-scope device array
// below, which the CUDA runtime places in every GPU that loads this library
// and keeps there until the process exits.  The caller passes only its input
// and output buffers (and, optionally, a word for the device status).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "rra.h"
#include "rra_internal.h"
#include "rra_static.h"

namespace {

constexpr int kMaxRanksStatic = RRA_STATIC_MAX_RANKS;                  // 8
constexpr size_t kMaxBytesStatic = RRA_STATIC_MAX_BYTES;               // 16 KiB per rank
constexpr size_t kSlotBytes = 2 * kMaxBytesStatic;                     // LL doubles every byte
constexpr size_t kParityBytes = (size_t)kMaxRanksStatic * kSlotBytes;  // one slot per source
constexpr size_t kWindowBytes = 2 * kParityBytes;                      // 512 KiB per window
constexpr size_t kCtrlBytes = (sizeof(rra::Ctrl) + 4095) / 4096 * 4096;
constexpr size_t kScratchBytes = kCtrlBytes + (size_t)kMaxRanksStatic * kWindowBytes;  // ~4.01 MiB
constexpr int kThreads = 256;
constexpr int kMaxDevices = 64;

// The scratch: control block (status word, epochs) followed by 8 windows of
// LL slots.  It is zero when the module loads, and all-zero is the idle
// state (status 0, epoch 1, LL flags 0), so no initialisation is needed --
// also not after cudaDeviceReset, when the module is loaded again.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceState {
    bool ready;
    char* base;          // device address of g_scratch on this device
    int sms;
    int blocks_per_sm[3];  // co-resident CTAs per SM of the LL one-shot kernel, per dtype
};

// Runs before every call's AllReduce, on its stream.  After a call that
// failed (a wait ran out: the status word is set), some CTAs may have left
// their epoch slots behind and LL flags of that epoch in the windows, so the
// whole array goes back to the idle state; otherwise it does nothing.  One
// CTA, so the status word is read and cleared by the same block.
__global__ void __launch_bounds__(1024) static_recover_kernel() {
    rra::Ctrl* ctrl = (rra::Ctrl*)g_scratch;
    __shared__ uint32_t failed;
    if (threadIdx.x == 0) failed = *(volatile uint32_t*)&ctrl->status;
    __syncthreads();
    if (failed == 0u) return;
    uint4* words = (uint4*)g_scratch;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (size_t i = threadIdx.x; i < kScratchBytes / sizeof(uint4); i += blockDim.x) words[i] = z;
}

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

size_t elem_size(rra_dtype_t d) { return d == RRA_FP32 ? 4 : d == RRA_BF16 ? 2 : d == RRA_FP64 ? 8 : 0; }

// Once per device, with that device current: look up the array's device
// address (cudaGetSymbolAddress) and query occupancy.  The address is looked
// up again on every call (host-side only, nothing is enqueued); if it moved
// -- the device was reset and the module loaded again -- the set-up is
// redone.  Set-up enqueues no work and does not synchronise.
rra_status_t setup(int dev, DeviceState** out) {
    std::lock_guard<std::mutex> g(g_mu);
    DeviceState& d = g_dev[dev];
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    if (!d.ready || d.base != (char*)ptr) {
        d.ready = false;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return RRA_ERR_CUDA;
        for (int t = 0; t < 3; ++t) {
            if (rra::occupancy((rra_dtype_t)t, rra::kKindOneshotLL, kThreads, &d.blocks_per_sm[t]) != cudaSuccess)
                return RRA_ERR_CUDA;
        }
        d.base = (char*)ptr;
        d.ready = true;
    }
    *out = &d;
    return RRA_OK;
}

}  // namespace

extern "C" rra_status_t rra_allreduce_static(int nranks, const void* const send[], void* const recv[],
                                             size_t count, rra_dtype_t dtype, uint32_t* dev_status,
                                             rra_stream_t stream) {
    if (nranks < 2 || nranks > kMaxRanksStatic || send == nullptr || recv == nullptr) return RRA_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (es == 0) return RRA_ERR_INVALID_ARG;
    if (count == 0) return RRA_OK;
    if (count > kMaxBytesStatic / es) return RRA_ERR_INVALID_ARG;  // larger than the static slots
    rra::Params p = {};
    for (int r = 0; r < nranks; ++r) {
        if (send[r] == nullptr || recv[r] == nullptr) return RRA_ERR_INVALID_ARG;
        if (((uintptr_t)send[r] | (uintptr_t)recv[r]) & 15u) return RRA_ERR_INVALID_ARG;
        p.send[r] = send[r];
        p.recv[r] = recv[r];
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RRA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RRA_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    rra_status_t st = setup(dev, &d);
    if (st != RRA_OK) return st;

    const size_t ve = rra::kVecBytes / es;
    const uint32_t nvec = (uint32_t)((count + ve - 1) / ve);
    int ctas = (int)((nvec + kThreads - 1) / kThreads);
    const int cmax = d->blocks_per_sm[dtype] * d->sms / nranks;
    if (cmax < 1) return RRA_ERR_NOT_CORESIDENT;
    if (ctas > cmax) ctas = cmax;
    p.win0 = d->base + kCtrlBytes;
    p.ctrl = (rra::Ctrl*)d->base;
    p.timing = nullptr;
    p.stride = kWindowBytes;
    p.count = count;
    p.timeout_ns = 1000000000ull;
    p.region_off = 0;
    p.slot_bytes = kSlotBytes;
    p.parity_bytes = kParityBytes;
    p.ll_off = 0;
    p.ll_bytes = kWindowBytes;
    p.llag_off = 0;
    p.llag_bytes = 0;
    p.nvec = nvec;
    p.chunk_vecs = nvec;  // one step: the message fits one slot
    p.per_cta = (nvec + (uint32_t)ctas - 1) / (uint32_t)ctas;
    p.ctas_per_rank = (int32_t)((nvec + p.per_cta - 1) / p.per_cta);
    p.nsteps = 1;
    p.nranks = nranks;
    p.epoch_slots = rra::kEpochSlots;
    p.drop_rank = -1;
    p.scrub_ranks = kMaxRanksStatic;  // calls with any rank count share the 8 windows

    cudaStream_t s = (cudaStream_t)stream;
    // The array keeps the previous call's contents.  After a successful call
    // that is the idle state of the next epoch (LL flags need no clearing:
    // each call uses new epochs); after a failed one, the recovery kernel
    // returns the whole array to the idle state first.
    static_recover_kernel<<<1, 1024, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess) return RRA_ERR_CUDA;
    const cudaError_t e = rra::launch_allreduce(p, dtype, rra::kKindOneshotLL, kThreads, s, true);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorCooperativeLaunchTooLarge ? RRA_ERR_NOT_CORESIDENT : RRA_ERR_CUDA;
    }
    if (dev_status != nullptr &&
        cudaMemcpyAsync(dev_status, &p.ctrl->status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return RRA_ERR_CUDA;
    return RRA_OK;
}
