// rra_static.cu -- an AllReduce entry point that allocates no device memory.
//
// Who needs it.  Some callers cannot call cudaMalloc at the moment they need
// an AllReduce, and cannot hold a communicator whose creation allocated for
// them either:
//  * code that runs while some other component is capturing a CUDA graph on
//    the device in the global capture mode, where cudaMalloc is refused;
//  * plug-ins and extensions whose host framework owns the GPU allocator and
//    forbids direct cudaMalloc / cudaFree (all device memory must come from
//    the framework, and the plug-in is only handed input and output buffers);
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
// LL slots.  Zero at load; set-up writes the idle state (epoch 1).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceState {
    bool ready;
    char* base;          // device address of g_scratch on this device
    int sms;
    int blocks_per_sm[3];  // co-resident CTAs per SM of the LL one-shot kernel, per dtype
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

size_t elem_size(rra_dtype_t d) { return d == RRA_FP32 ? 4 : d == RRA_BF16 ? 2 : d == RRA_FP64 ? 8 : 0; }

// Once per device, with that device current: look up the array's device
// address, query occupancy, and write the idle state (epoch 1, LL flags 0,
// status 0, no injected fault).  Synchronises the device, so the first call
// on a device must not happen while a stream is being captured.
rra_status_t setup(int dev, DeviceState** out) {
    std::lock_guard<std::mutex> g(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return RRA_ERR_CUDA;
        }
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return RRA_ERR_CUDA;
        for (int t = 0; t < 3; ++t) {
            if (rra::occupancy((rra_dtype_t)t, rra::kKindOneshotLL, kThreads, &d.blocks_per_sm[t]) != cudaSuccess)
                return RRA_ERR_CUDA;
        }
        rra_layout_t lay = {};
        lay.nranks = kMaxRanksStatic;
        lay.ll_bytes = kWindowBytes;
        lay.window_stride = kWindowBytes;
        lay.ctrl_bytes = kCtrlBytes;
        lay.total_bytes = kScratchBytes;
        if (rra::launch_init((char*)ptr, kScratchBytes, lay, kMaxRanksStatic, 0) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
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

    cudaStream_t s = (cudaStream_t)stream;
    // The array keeps the previous call's contents.  The status word must start
    // at zero (a failed earlier call would otherwise turn this one into a
    // no-op); LL flags need no clearing (each call uses new epochs).
    if (cudaMemsetAsync(&p.ctrl->status, 0, sizeof(uint32_t), s) != cudaSuccess) return RRA_ERR_CUDA;
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
