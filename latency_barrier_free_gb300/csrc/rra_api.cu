// rra_api.cu -- host side of the C ABI declared in include/rra.h.
//
// The communicator owns one device allocation: a control block followed by N
// windows at a fixed stride ("symmetric memory", "Every Microsecond Matters"
// Sec. II-B, restated for virtual ranks on one GPU).  Window regions, in
// order: one-shot LL slots, one-shot sentinel slots, two-shot RS + AG slots,
// LL128-atomic accumulators + counters + LL AllGather slots.  Scratch caps
// default to the paper's sizes (Sec. VII, Fig. 12): 4 MiB per window for
// one-shot, 64 MiB for two-shot and LL128-atomic; messages larger than a
// step's capacity run as a chunk loop (Sec. IV, double buffering).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <array>
#include <map>
#include <mutex>

#include "rra.h"
#include "rra_internal.h"
#include "placement.h"

static_assert(rra::placement::kMaxRanks == RRA_MAX_RANKS, "bulk-copy kernels serve every rank count");
static_assert(rra::placement::kVecBytes == (size_t)rra::kVecBytes, "one transfer vector");

using rra::Ctrl;
using rra::Params;

namespace {

constexpr size_t kDefaultScratchOneshot = 4ull << 20;   // Fig. 12: one-shot
constexpr size_t kDefaultScratchTwoshot = 64ull << 20;  // Fig. 12: two-shot, LL128
constexpr size_t kWindowAlign = 64ull << 10;
// Default two-shot / LL128 step size: keep the scratch live in one step (all
// windows, both parities) near this size, so it stays in L2 while the
// inputs and outputs stream through HBM (measured on GB300: a 64 MiB cap's
// 16 MiB steps spilled scratch to DRAM, 2.3x the compulsory traffic).
constexpr size_t kLiveScratch = 32ull << 20;
// The LL128-atomic's step keeps about twice that live (accumulators, counters
// and LL AllGather slots of all windows): its scratch is touched by atomics
// and polls rather than streamed, and a 64 MiB step measured equal or faster
// at N = 8..64 (N = 64, 256 KiB per rank: one step of 512 CTAs in 35 us
// against two steps of 256 CTAs in 51 us).
constexpr size_t kLiveScratchLL128 = 64ull << 20;

size_t floor16(size_t x) { return x & ~(size_t)15; }
size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }
size_t align_up(size_t x, size_t a) { return ceil_div(x, a) * a; }

size_t elem_size(rra_dtype_t d) {
    switch (d) {
        case RRA_FP32: return 4;
        case RRA_BF16: return 2;
        case RRA_FP64: return 8;
    }
    return 0;
}

bool valid_algo(int a) { return a >= RRA_ONESHOT_LL && a <= RRA_TWOSHOT_BARRIER; }
bool is_cluster(int a) { return a == RRA_ONESHOT_CLUSTER || a == RRA_TWOSHOT_CLUSTER; }
bool valid_dtype(int d) { return d >= RRA_FP32 && d <= RRA_FP64; }

int64_t env_i64(const char* name, int64_t dflt) {
    const char* s = getenv(name);
    if (s == nullptr || *s == '\0') return dflt;
    char* end = nullptr;
    long long v = strtoll(s, &end, 10);
    if (end == s) return dflt;
    return (int64_t)v;
}

// LL128-atomic region of one window for a partition of `part` payload bytes.
struct LaSizes {
    size_t acc_parity;   // accumulator bytes per parity (bf16 needs 2x: binary32 accumulators)
    size_t cnt_parity;   // counter bytes per parity
    size_t ag_slot;      // LL AllGather slot bytes (2x payload)
    size_t total;
};
LaSizes la_sizes(size_t part, int n) {
    LaSizes s;
    s.acc_parity = 2 * part;
    const size_t groups = ceil_div(part / rra::kVecBytes, rra::kGroupVecs);
    s.cnt_parity = align_up(groups * 4, 256);
    s.ag_slot = 2 * part;
    s.total = 2 * s.acc_parity + 2 * s.cnt_parity + 2 * (size_t)n * s.ag_slot;
    return s;
}

}  // namespace

struct rra_comm {
    int device = -1;
    int nranks = 0;
    size_t max_bytes = 0;
    size_t cap_oneshot = 0, cap_twoshot = 0;
    rra_layout_t lay = {};
    char* base = nullptr;
    Ctrl* ctrl = nullptr;
    char* win0 = nullptr;
    int sm_count = 0;
    int threads = 128;
    bool threads_set = false;              // THREADS given by the user (attribute or environment)
    int64_t ctas_per_rank = 0;
    int64_t timeout_ms = 1000;
    int64_t ts_chunk = 0, la_chunk = 0, os_chunk = 0;
    int blocks_per_sm[3][rra::kNumKinds];  // by dtype, kernel kind; -1 = not queried
    int64_t oneshot_wide = -1;              // -1 auto (N >= 16), 0 never, 1 always
    int64_t cooperative = 1;                // cooperative launch (co-residency guaranteed)
    int64_t pdl = 1;                        // programmatic dependent launch
    int64_t cluster_slice = 0;              // cluster kernels: bytes per rank per slice, 0 = auto
    int64_t cluster_pipe = 0;               // persistent cluster two-shot: -1 auto, 0 never (default), 1 always
    int64_t cluster_tma = -1;               // cluster one-/two-shot push by bulk copies: -1 auto (default), 0, 1
    int64_t host_zero_copy = 1;             // rra_allreduce_host: run on mapped pinned buffers directly
    int cluster_fits[2][3] = {{-1, -1, -1}, {-1, -1, -1}};  // [two-shot][dtype]: -1 not queried
    int cluster_multi_fits[2][2][3] = {{{-1, -1, -1}, {-1, -1, -1}}, {{-1, -1, -1}, {-1, -1, -1}}};
                                            // the same for N > 16: [bulk-copy push][two-shot][dtype]
    std::map<uint64_t, int> cluster_waves;  // (dtype, threads, stage bytes) -> clusters resident at once
    int coll_fits[2][6][3] = {{{-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}},
                              {{-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}, {-1, -1, -1}}};
                              // [bulk-copy kernel][op][dtype]
    int64_t coll_split = -1;                // Broadcast/Reduce in two hops: -1 auto, 0 never, 1 always
    int residual_fits[2][2][3] = {{{-1, -1, -1}, {-1, -1, -1}}, {{-1, -1, -1}, {-1, -1, -1}}};  // [bulk][two][dtype]
    int residual_multi_fits[2][3] = {{-1, -1, -1}, {-1, -1, -1}};  // the same for N > 16
    rra::placement::SourceCache local_sources;  // source sets that passed the bulk-copy check
    const char* last_kernel = "none";       // the kernel the last enqueued call launched
    int32_t drop_rank = -1;                 // injected fault (rra_comm_inject_drop), -1 = none
    bool poisoned = false;
    uint64_t* timing = nullptr;
    uint64_t* trace = nullptr;
    // rra_allreduce_host staging (allocated on first use)
    char* stage = nullptr;
    size_t stage_slot = 0;
    uint32_t* host_status = nullptr;       // pinned host word (device-mapped when host_mirror)
    bool host_mirror = false;              // device code mirrors the status word into host_status
    std::mutex mu;
};

// ----------------------------------------------------------------------------
// Where the bulk-copy push may run.  Its copies (cp.async.bulk ...
// .multicast::cluster, issued by cluster_tma_kernel, coll_bulk_kernel and the
// device API's bulk sends) read straight from the caller's buffers.  They are
// issued only when every buffer they read is device memory of the
// communicator's own GPU -- checked at both ends of the range a copy reads --
// and the process holds no context on another GPU.  Any other call (host
// memory, another GPU's memory, managed memory, or a process that also
// drives other GPUs) pushes with st.async stores instead: the same results.

namespace {

// cuDevicePrimaryCtxGetState / cuDeviceGet, looked up once through the
// runtime (no link against the driver library).
typedef int (*PfnPrimaryCtxGetState)(int dev, unsigned int* flags, int* active);
typedef int (*PfnDeviceGet)(int* dev, int ordinal);

// True when the process holds an active primary context on a GPU other
// than `dev`, or when that cannot be determined.
bool other_gpu_in_use(int dev) {
    static std::once_flag once;
    static int ndev = -1;
    static PfnPrimaryCtxGetState ctx_state = nullptr;
    static PfnDeviceGet device_get = nullptr;
    std::call_once(once, [] {
        int n = 0;
        if (cudaGetDeviceCount(&n) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        ndev = n;
        if (n <= 1) return;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuDevicePrimaryCtxGetState", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            ctx_state = (PfnPrimaryCtxGetState)f;
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuDeviceGet", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            device_get = (PfnDeviceGet)f;
        cudaGetLastError();
    });
    if (ndev < 0) return true;
    if (ndev <= 1) return false;
    if (ctx_state == nullptr || device_get == nullptr) return true;
    for (int d = 0; d < ndev; ++d) {
        if (d == dev) continue;
        int h = 0, active = 0;
        unsigned int flags = 0;
        if (device_get(&h, d) != 0 || ctx_state(h, &flags, &active) != 0) return true;
        if (active) return true;
    }
    return false;
}

// True when address `p` lies in device memory of GPU `dev`.
bool on_device(int dev, const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

}  // namespace

// True when bulk copies may read `bytes` from each of src[0..n-1] (the rule
// and its cache: placement.h).  Called with c->mu held.
static bool bulk_sources_local(rra_comm* c, const void* const src[], int n, size_t bytes) {
    const int dev = c->device;
    return rra::placement::bulk_sources_local(c->local_sources, other_gpu_in_use(dev), src, n, bytes,
                                              [dev](const void* p) { return on_device(dev, p); });
}

extern "C" {

const char* rra_version(void) { return "0.1.0"; }

const char* rra_status_string(rra_status_t s) {
    switch (s) {
        case RRA_OK: return "ok";
        case RRA_ERR_INVALID_ARG: return "invalid argument";
        case RRA_ERR_CUDA: return "CUDA runtime error";
        case RRA_ERR_OOM: return "out of device memory";
        case RRA_ERR_NOT_CORESIDENT: return "ranks cannot all be co-resident on the GPU";
        case RRA_ERR_TIMEOUT: return "a device-side wait timed out";
        case RRA_ERR_POISONED: return "communicator poisoned by an earlier device error; reset it";
    }
    return "unknown status";
}

// Choice without the cluster kernels (also the fallback when the device
// cannot schedule a cluster of N CTAs).
static rra_algo_t select_global(int nranks, size_t bytes) {
    const size_t total = (size_t)nranks * bytes;
    if (nranks <= 8) return total <= (3ull << 19) ? RRA_ONESHOT_SENTINEL : RRA_TWOSHOT_DIRECT;
    const size_t ll128_max = nranks >= 64 ? (64u << 10) : (16u << 10);
    if (bytes <= (4u << 10)) return RRA_ONESHOT_SENTINEL;
    if (bytes <= ll128_max) return RRA_LL128_ATOMIC;
    return RRA_TWOSHOT_DIRECT;
}

// The cluster one-shot / two-shot crossover, measured on GB300 with CUDA-graph
// replay (N = 2..64).  With the bulk-copy push, up to 16 ranks the one-shot
// while N^2 M <= 8 MiB at N <= 2, 2 MiB at N <= 4, 4 MiB at N <= 8, 8 MiB
// above, and above 16 ranks while 16 N M <= 16 MiB (N = 20, 32, 64: the
// one-shot faster up to 16 KiB per rank, the two-shot from 64 KiB); with
// st.async pushes (the bulk-copy push off) while min(N, 16) N M <= 1 MiB.
static rra_algo_t select_cluster(int nranks, size_t bytes, bool bulk_copy) {
    const size_t n = (size_t)nranks;
    if (nranks <= rra::kClusterMaxRanks && bulk_copy) {
        const size_t limit = (n <= 2 ? 8ull : n <= 4 ? 2ull : n <= 8 ? 4ull : 8ull) << 20;
        return n * n * bytes <= limit ? RRA_ONESHOT_CLUSTER : RRA_TWOSHOT_CLUSTER;
    }
    const size_t g = std::min<size_t>(n, rra::kClusterMaxRanks);
    const size_t limit = bulk_copy ? (16ull << 20) : (1ull << 20);
    return g * n * bytes <= limit ? RRA_ONESHOT_CLUSTER : RRA_TWOSHOT_CLUSTER;
}

// Whether a cluster call pushes by bulk copies: unless the attribute turns
// it off (it measured faster at every N = 2..16 and every size from 128 B
// to 64 MiB on GB300, and above 16 ranks as well).
static bool bulk_copy_push(const rra_comm* c) {
    return c->cluster_tma != 0;
}

rra_status_t rra_select_algo(int nranks, size_t bytes, rra_dtype_t dtype, rra_algo_t* out) {
    if (out == nullptr || nranks < 2 || nranks > RRA_MAX_RANKS || !valid_dtype(dtype)) return RRA_ERR_INVALID_ARG;
    *out = select_cluster(nranks, bytes, true);  // the default attributes: bulk-copy push on
    return RRA_OK;
}

rra_status_t rra_plan_layout(int nranks, size_t max_bytes, size_t scratch_oneshot,
                             size_t scratch_twoshot, rra_layout_t* out) {
    if (out == nullptr || nranks < 2 || nranks > RRA_MAX_RANKS || max_bytes == 0)
        return RRA_ERR_INVALID_ARG;
    if (max_bytes > rra::kMaxMessageBytes) return RRA_ERR_INVALID_ARG;
    const size_t cap_os = scratch_oneshot ? scratch_oneshot : kDefaultScratchOneshot;
    const size_t cap_ts = scratch_twoshot ? scratch_twoshot : kDefaultScratchTwoshot;
    const size_t n = (size_t)nranks;
    const size_t nvec = ceil_div(max_bytes, rra::kVecBytes);
    const size_t payload = nvec * rra::kVecBytes;
    const size_t part_need = ceil_div(nvec, n) * rra::kVecBytes;

    rra_layout_t L = {};
    L.nranks = nranks;
    L.max_bytes = max_bytes;
    // One-shot: 2 parities x N source slots; LL doubles every payload byte
    // (Fig. 8: 2 x sizeof(T) per element in LL mode).
    L.ll_chunk = std::min(payload, floor16(cap_os / (2 * n * 2)));
    L.os_chunk = std::min(payload, floor16(cap_os / (2 * n)));
    // Two-shot: RS and AG regions, each 2 parities x N slots of one partition.
    L.ts_part = std::min(part_need, floor16(cap_ts / (4 * n)));
    // LL128-atomic: shrink the partition until the region fits the cap.
    size_t la_part = std::min(part_need, floor16(cap_ts / (4 * (n + 1))));
    while (la_part >= (size_t)rra::kVecBytes && la_sizes(la_part, nranks).total > cap_ts)
        la_part -= rra::kVecBytes;
    L.la_part = la_part;
    if (L.ll_chunk < 16 || L.os_chunk < 16 || L.ts_part < 16 || L.la_part < 16)
        return RRA_ERR_INVALID_ARG;
    // Barrier baseline: one parity (the second barrier frees the buffers).
    L.bd_chunk = std::min(payload, floor16(cap_os / n));
    if (L.bd_chunk < 16) return RRA_ERR_INVALID_ARG;
    L.ll_bytes = align_up(2 * n * 2 * L.ll_chunk, rra::kRegionAlign);
    L.bf_bytes = align_up((size_t)rra::kBarrierCtas * RRA_MAX_RANKS * 4, rra::kRegionAlign);
    L.os_bytes = align_up(2 * n * L.os_chunk, rra::kRegionAlign);
    L.ts_bytes = align_up(2 * (2 * n * L.ts_part), rra::kRegionAlign);
    L.la_bytes = align_up(la_sizes(L.la_part, nranks).total, rra::kRegionAlign);
    L.bd_bytes = align_up(2 * n * L.bd_chunk, rra::kRegionAlign);  // slots; the two-shot baseline's AllGather
    L.window_stride = align_up(L.ll_bytes + L.bf_bytes + L.os_bytes + L.ts_bytes + L.la_bytes + L.bd_bytes,
                               kWindowAlign);
    L.ctrl_bytes = align_up(sizeof(Ctrl), rra::kRegionAlign);
    L.total_bytes = L.ctrl_bytes + n * L.window_stride;
    *out = L;
    return RRA_OK;
}

// Largest CTA a kernel kind is built for: the two-shot kernels are built for
// 4 CTAs of 128 threads per SM, the others for up to 256 threads.
static int kind_max_threads(int kind) {
    return kind == rra::kKindTwoshot || kind == rra::kKindTwoshotDirect ? 128 : 256;
}

static rra_status_t query_blocks(rra_comm* c, rra_dtype_t d, int kind, int* out) {
    int& b = c->blocks_per_sm[d][kind];
    if (b < 0) {
        int v = 0;
        if (rra::occupancy(d, kind, std::min(c->threads, kind_max_threads(kind)), &v) != cudaSuccess)
            return RRA_ERR_CUDA;
        b = v;
    }
    *out = b;
    return RRA_OK;
}

rra_status_t rra_comm_create(int nranks, size_t max_bytes, rra_comm_t* out) {
    if (out == nullptr) return RRA_ERR_INVALID_ARG;
    const size_t cap_os = (size_t)std::max<int64_t>(0, env_i64("RRA_SCRATCH_ONESHOT", 0));
    const size_t cap_ts = (size_t)std::max<int64_t>(0, env_i64("RRA_SCRATCH_TWOSHOT", 0));
    rra_layout_t lay;
    rra_status_t st = rra_plan_layout(nranks, max_bytes, cap_os, cap_ts, &lay);
    if (st != RRA_OK) return st;

    rra_comm* c = new (std::nothrow) rra_comm();
    if (c == nullptr) return RRA_ERR_OOM;
    c->nranks = nranks;
    c->max_bytes = max_bytes;
    c->cap_oneshot = cap_os;
    c->cap_twoshot = cap_ts;
    c->lay = lay;
    for (auto& row : c->blocks_per_sm)
        for (int& b : row) b = -1;
    c->timeout_ms = env_i64("RRA_POLL_TIMEOUT_MS", 1000);
    c->ctas_per_rank = env_i64("RRA_CTAS_PER_RANK", 0);
    const int64_t thr = env_i64("RRA_THREADS", 128);
    if (thr == 64 || thr == 128 || thr == 256) c->threads = (int)thr;
    c->threads_set = getenv("RRA_THREADS") != nullptr;
    if (c->timeout_ms <= 0) c->timeout_ms = 1000;
    if (c->ctas_per_rank < 0) c->ctas_per_rank = 0;

    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
        delete c;
        return RRA_ERR_CUDA;
    }
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device) != cudaSuccess || !coop) {
        delete c;
        return RRA_ERR_CUDA;
    }
    // Every kernel must fit at least one CTA per rank at once.
    for (int d = 0; d < 3; ++d) {
        for (int a = 0; a < rra::kNumKinds; ++a) {
            int b = 0;
            if (query_blocks(c, (rra_dtype_t)d, a, &b) != RRA_OK) {
                delete c;
                return RRA_ERR_CUDA;
            }
            if ((int64_t)b * c->sm_count < nranks) {
                delete c;
                return RRA_ERR_NOT_CORESIDENT;
            }
        }
    }
    if (cudaMalloc((void**)&c->base, lay.total_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return RRA_ERR_OOM;
    }
    c->ctrl = (Ctrl*)c->base;
    c->win0 = c->base + lay.ctrl_bytes;
    // A pinned, device-mapped host word that device code writes together with
    // the status word on the first error: the host entry reads it after
    // synchronising instead of copying the status word back.
    uint32_t* mirror_dev = nullptr;
    if (cudaHostAlloc((void**)&c->host_status, sizeof(uint32_t), cudaHostAllocMapped) == cudaSuccess) {
        *c->host_status = 0u;
        if (cudaHostGetDevicePointer((void**)&mirror_dev, c->host_status, 0) != cudaSuccess) mirror_dev = nullptr;
    } else {
        c->host_status = nullptr;
    }
    cudaGetLastError();
    if (rra::launch_init(c->base, lay.total_bytes, lay, nranks, 0) != cudaSuccess ||
        cudaMemcpy(&c->ctrl->host_status, &mirror_dev, sizeof(mirror_dev), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(c->base);
        if (c->host_status) cudaFreeHost(c->host_status);
        delete c;
        return RRA_ERR_CUDA;
    }
    c->host_mirror = mirror_dev != nullptr;
    *out = c;
    return RRA_OK;
}

rra_status_t rra_comm_destroy(rra_comm_t c) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    rra_status_t st = RRA_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) st = RRA_ERR_CUDA;
    if (c->base) cudaFree(c->base);
    if (c->stage) cudaFree(c->stage);
    if (c->host_status) cudaFreeHost(c->host_status);
    delete c;
    return st;
}

rra_status_t rra_comm_layout(rra_comm_t c, rra_layout_t* out) {
    if (c == nullptr || out == nullptr) return RRA_ERR_INVALID_ARG;
    *out = c->lay;
    return RRA_OK;
}

rra_status_t rra_comm_set_attr(rra_comm_t c, rra_attr_t attr, int64_t v) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(c->mu);
    switch (attr) {
        case RRA_ATTR_CTAS_PER_RANK:
            if (v < 0 || v > rra::kEpochSlots) return RRA_ERR_INVALID_ARG;
            c->ctas_per_rank = v;
            return RRA_OK;
        case RRA_ATTR_POLL_TIMEOUT_MS:
            if (v <= 0 || v > 3600000) return RRA_ERR_INVALID_ARG;
            c->timeout_ms = v;
            return RRA_OK;
        case RRA_ATTR_THREADS:
            if (v != 64 && v != 128 && v != 256) return RRA_ERR_INVALID_ARG;
            if (c->threads != (int)v) {
                c->threads = (int)v;
                c->threads_set = true;
                for (auto& row : c->blocks_per_sm)
                    for (int& b : row) b = -1;
            }
            return RRA_OK;
        case RRA_ATTR_TWOSHOT_CHUNK:
            if (v < 0 || v % 16) return RRA_ERR_INVALID_ARG;
            c->ts_chunk = v;
            return RRA_OK;
        case RRA_ATTR_LL128_CHUNK:
            if (v < 0 || v % 16) return RRA_ERR_INVALID_ARG;
            c->la_chunk = v;
            return RRA_OK;
        case RRA_ATTR_ONESHOT_CHUNK:
            if (v < 0 || v % 16) return RRA_ERR_INVALID_ARG;
            c->os_chunk = v;
            return RRA_OK;
        case RRA_ATTR_ONESHOT_WIDE:
            if (v < -1 || v > 1) return RRA_ERR_INVALID_ARG;
            c->oneshot_wide = v;
            return RRA_OK;
        case RRA_ATTR_COOPERATIVE:
            if (v < 0 || v > 1) return RRA_ERR_INVALID_ARG;
            c->cooperative = v;
            return RRA_OK;
        case RRA_ATTR_PDL:
            if (v < 0 || v > 1) return RRA_ERR_INVALID_ARG;
            c->pdl = v;
            return RRA_OK;
        case RRA_ATTR_CLUSTER_SLICE:
            if (v < 0 || v % 16 || v > (int64_t)rra::kClusterStageBytes) return RRA_ERR_INVALID_ARG;
            c->cluster_slice = v;
            return RRA_OK;
        case RRA_ATTR_CLUSTER_PIPE:
            if (v < -1 || v > 1) return RRA_ERR_INVALID_ARG;
            c->cluster_pipe = v;
            return RRA_OK;
        case RRA_ATTR_HOST_ZERO_COPY:
            if (v < 0 || v > 1) return RRA_ERR_INVALID_ARG;
            c->host_zero_copy = v;
            return RRA_OK;
        case RRA_ATTR_COLL_SPLIT:
            if (v < -1 || v > 1) return RRA_ERR_INVALID_ARG;
            c->coll_split = v;
            return RRA_OK;
        case RRA_ATTR_CLUSTER_TMA:
            if (v < -1 || v > 1) return RRA_ERR_INVALID_ARG;
            c->cluster_tma = v;
            return RRA_OK;
    }
    return RRA_ERR_INVALID_ARG;
}

rra_status_t rra_comm_get_attr(rra_comm_t c, rra_attr_t attr, int64_t* v) {
    if (c == nullptr || v == nullptr) return RRA_ERR_INVALID_ARG;
    switch (attr) {
        case RRA_ATTR_CTAS_PER_RANK: *v = c->ctas_per_rank; return RRA_OK;
        case RRA_ATTR_POLL_TIMEOUT_MS: *v = c->timeout_ms; return RRA_OK;
        case RRA_ATTR_THREADS: *v = c->threads; return RRA_OK;
        case RRA_ATTR_TWOSHOT_CHUNK: *v = c->ts_chunk; return RRA_OK;
        case RRA_ATTR_LL128_CHUNK: *v = c->la_chunk; return RRA_OK;
        case RRA_ATTR_ONESHOT_CHUNK: *v = c->os_chunk; return RRA_OK;
        case RRA_ATTR_ONESHOT_WIDE: *v = c->oneshot_wide; return RRA_OK;
        case RRA_ATTR_COOPERATIVE: *v = c->cooperative; return RRA_OK;
        case RRA_ATTR_PDL: *v = c->pdl; return RRA_OK;
        case RRA_ATTR_CLUSTER_SLICE: *v = c->cluster_slice; return RRA_OK;
        case RRA_ATTR_CLUSTER_PIPE: *v = c->cluster_pipe; return RRA_OK;
        case RRA_ATTR_HOST_ZERO_COPY: *v = c->host_zero_copy; return RRA_OK;
        case RRA_ATTR_COLL_SPLIT: *v = c->coll_split; return RRA_OK;
        case RRA_ATTR_CLUSTER_TMA: *v = c->cluster_tma; return RRA_OK;
    }
    return RRA_ERR_INVALID_ARG;
}

// More ranks than a cluster holds (N > 16): clusters of 16 CTAs, CTA j
// hosting ranks j, j + 16, ...; one cluster per slice of S vectors.  A
// window holds N slots: N x S vectors (one-shot) or N x S/16 (two-shot, S a
// multiple of 16) within the 96 KiB stage.  S: the whole message while it
// fits one slice (one-shot) or, for the two-shot, about two CTAs per SM.
static rra_status_t plan_cluster_multi(rra_comm* c, size_t count, rra_dtype_t dtype, bool two, Params* p,
                                       int* threads, int* mode, bool bulk) {
    const size_t n = (size_t)c->nranks;
    const size_t g = (size_t)rra::kClusterMaxRanks;
    const int kmode = bulk ? (two ? rra::kClusterTwoshotMultiTma : rra::kClusterOneshotMultiTma)
                           : (two ? rra::kClusterTwoshotMulti : rra::kClusterOneshotMulti);
    int& fits = c->cluster_multi_fits[bulk ? 1 : 0][two ? 1 : 0][(int)dtype];
    if (fits < 0) fits = rra::cluster_max_active(dtype, kmode, c->nranks, 256, rra::kClusterStageBytes) > 0 ? 1 : 0;
    if (fits == 0) return RRA_ERR_NOT_CORESIDENT;
    const size_t ve = rra::kVecBytes / elem_size(dtype);
    memset(p, 0, sizeof(*p));
    p->win0 = c->win0;
    p->ctrl = c->ctrl;
    p->timing = c->timing;
    p->trace = c->trace;
    p->stride = c->lay.window_stride;
    p->count = count;
    p->nvec = (uint32_t)ceil_div(count, ve);
    p->timeout_ns = (uint64_t)c->timeout_ms * 1000000ull;
    p->nranks = c->nranks;
    p->nsteps = 1;
    p->chunk_vecs = p->nvec;
    p->epoch_slots = rra::kEpochSlots;
    const size_t stage_vecs = rra::kClusterStageBytes / rra::kVecBytes;
    const size_t smax = two ? (stage_vecs / n) * g : stage_vecs / n;  // N x S (one-shot), N x S/16 (two-shot)
    size_t S;
    if (c->cluster_slice > 0) {
        S = (size_t)c->cluster_slice / rra::kVecBytes;
    } else if (two) {
        const size_t target = std::max<size_t>(1, 2 * (size_t)c->sm_count / g);
        S = std::max<size_t>(g, ceil_div(p->nvec, target));
    } else {
        S = p->nvec;
    }
    if (two) S = align_up(S, g);
    S = std::max<size_t>(two ? g : 1, std::min(S, smax));
    p->per_cta = (uint32_t)S;
    p->ctas_per_rank = (int32_t)ceil_div(p->nvec, S);  // clusters (slices)
    const size_t hosted = ceil_div(n, g);
    const size_t cap = c->threads_set ? (size_t)c->threads : 256;
    *threads = (int)std::min<size_t>(cap, std::max<size_t>(32, align_up(S * hosted, 32)));
    *mode = kmode;
    return RRA_OK;
}

// Plan of a cluster call: one cluster of N CTAs per slice of S vectors, CTA
// r of a cluster = rank r, the push made by bulk copies (cluster_tma_kernel)
// unless RRA_ATTR_CLUSTER_TMA is 0 or the persistent two-shot is asked for.
// S: for the bulk-copy two-shot up to N M = 4 MiB on device buffers,
// partitions of 64 vectors; otherwise one position per thread while the
// message is small, then about two CTAs per SM in one wave, up to one batch
// of kClusterBatch loads per thread (GB300 sweep: 16 KiB slices of 128
// threads were fastest from 4 MiB up at N = 2..16); at most the 96 KiB stage
// (N x S vectors for the one-shot, S for the two-shot, whose S is a multiple
// of N).
//
// With RRA_ATTR_CLUSTER_PIPE (off by default) the two-shot runs on the
// persistent, double-buffered kernel: as many clusters as can be resident,
// each looping over its share of the slices.
// host: the buffers are pinned host memory (read and written over
// NVLink-C2C), where larger copies measured faster.  local: every input is
// device memory of this GPU (bulk_sources_local); only then may the push be
// made by bulk copies.
static rra_status_t plan_cluster(rra_comm* c, size_t count, rra_dtype_t dtype, rra_algo_t algo, Params* p,
                                 int* threads, int* mode, bool host, bool local) {
    const bool two = algo == RRA_TWOSHOT_CLUSTER;
    const size_t n = (size_t)c->nranks;
    if (c->nranks > rra::kClusterMaxRanks)
        return plan_cluster_multi(c, count, dtype, two, p, threads, mode, bulk_copy_push(c) && local && !host);
    int& fits = c->cluster_fits[two ? 1 : 0][(int)dtype];
    if (fits < 0)
        fits = rra::cluster_max_active(dtype, two ? rra::kClusterTwoshot : rra::kClusterOneshot, c->nranks, 256,
                                       rra::kClusterStageBytes) > 0
                   ? 1
                   : 0;
    if (fits == 0) return RRA_ERR_NOT_CORESIDENT;
    const size_t ve = rra::kVecBytes / elem_size(dtype);
    memset(p, 0, sizeof(*p));
    p->win0 = c->win0;
    p->ctrl = c->ctrl;
    p->timing = c->timing;
    p->trace = c->trace;
    p->stride = c->lay.window_stride;
    p->count = count;
    p->nvec = (uint32_t)ceil_div(count, ve);
    p->timeout_ns = (uint64_t)c->timeout_ms * 1000000ull;
    p->nranks = c->nranks;
    p->nsteps = 1;
    p->chunk_vecs = p->nvec;
    const size_t stage_vecs = rra::kClusterStageBytes / rra::kVecBytes;
    const size_t smax = two ? stage_vecs / n * n : stage_vecs / n;
    size_t S;
    size_t T = (size_t)c->threads;
    const size_t s_mid = ceil_div((size_t)p->nvec * n, 512);  // ~512 CTAs in all
    const bool bulk = c->cluster_pipe == 0 && bulk_copy_push(c) && local && !host;
    if (c->cluster_slice > 0) {
        S = (size_t)c->cluster_slice / rra::kVecBytes;
    } else if (two && bulk && !host && n * p->nvec <= (256u << 10)) {
        // bulk-copy two-shot up to N M = 4 MiB: partitions of 64 vectors
        // (1 KiB copies), one reduced position per thread (GB300 sweep at
        // N = 4, 8, 16: 1 MiB at N = 4 in 2.85 us against 3.6 us with the
        // st.async-era shape below)
        if (!c->threads_set) T = n <= 8 ? 64 : 128;
        S = 64 * n;
    } else if (two && host) {
        // host buffers (zero copy): 4 KiB slices, 256 threads, one vector per
        // thread.  Every load crosses the host link, so more, smaller slices
        // keep more of it busy (GB300, N = 4: 4 MiB per rank in 106 us in the
        // kernel against 154 us with the device-memory shape below, at the
        // link's rate for reading and writing at once; 1 MiB 44 against 50 us
        // per synchronised call)
        if (!c->threads_set) T = 256;
        S = 256;
    } else if (two && s_mid <= 1024) {
        // two-shot up to ~1-2 MiB per rank (latency-bound): about 512 CTAs of
        // 256 threads, 2-4 vectors per thread (GB300 sweep at N = 4, 8:
        // 1 MiB in 3.5 / 5.5 us against 4.7 / 8.1 with the rule below)
        if (!c->threads_set) T = 256;
        S = std::max<size_t>(std::min<size_t>(p->nvec, T), s_mid);
    } else {
        // one vector per thread for small messages; then spread over about
        // two CTAs per SM, but at most one batch of loads per thread
        const size_t target = std::max<size_t>(1, 2 * (size_t)c->sm_count / n);
        S = std::max<size_t>(std::min<size_t>(p->nvec, T), ceil_div(p->nvec, target));
        S = std::min<size_t>(S, T * rra::kClusterBatch);
    }
    if (two) S = align_up(S, n);
    S = std::max<size_t>(two ? n : 1, std::min(S, smax));
    p->per_cta = (uint32_t)S;
    const size_t nslices = ceil_div(p->nvec, S);
    p->ctas_per_rank = (int32_t)nslices;  // one cluster per slice
    p->epoch_slots = rra::kEpochSlots;
    *threads = (int)std::min<size_t>(T, std::max<size_t>(32, align_up(S, 32)));
    *mode = two ? rra::kClusterTwoshot : rra::kClusterOneshot;
    // the persistent two-shot, when asked for, keeps its st.async pushes
    if (bulk) {
        *mode = two ? rra::kClusterTwoshotTma : rra::kClusterOneshotTma;
        return RRA_OK;
    }
    if (two && c->cluster_pipe != 0 && S <= (size_t)*threads * rra::kClusterBatch &&
        2 * S * rra::kVecBytes <= rra::kClusterStageBytes) {
        const size_t smem = 2 * S * rra::kVecBytes;
        const uint64_t key = ((uint64_t)dtype << 40) | ((uint64_t)*threads << 24) | (uint64_t)smem;
        auto it = c->cluster_waves.find(key);
        if (it == c->cluster_waves.end())
            it = c->cluster_waves
                     .emplace(key, rra::cluster_max_active(dtype, rra::kClusterTwoshotPipe, c->nranks, *threads, smem))
                     .first;
        const size_t wave = (size_t)it->second;
        if (wave > 0 && (nslices > wave || c->cluster_pipe == 1)) {
            // RRA_ATTR_CTAS_PER_RANK, when set, caps the number of clusters
            const size_t g = c->ctas_per_rank > 0 ? std::min(wave, (size_t)c->ctas_per_rank) : wave;
            *mode = rra::kClusterTwoshotPipe;
            p->ctas_per_rank = (int32_t)std::min(nslices, g);
            p->nsteps = (uint32_t)nslices;
        }
    }
    return RRA_OK;
}

// Plan of a ReduceScatter / AllGather / Broadcast / Reduce call: one cluster
// of N CTAs per slice of S vectors of a block of `count` elements; S as for
// the cluster AllReduce (one vector per thread while small, then about two
// CTAs per SM), with at most one batch of kClusterBatch input vectors per
// thread and the 96 KiB stage (N slots of S vectors; one slot for Broadcast).
static rra_status_t plan_coll(rra_comm* c, size_t count, rra_dtype_t dtype, int op, int root, bool bulk,
                              bool store_bulk, Params* p, int* threads) {
    int& fits = c->coll_fits[bulk ? 1 : 0][op][(int)dtype];
    if (fits < 0) fits = rra::coll_max_active(dtype, op, c->nranks, 256, rra::kClusterStageBytes, bulk) > 0 ? 1 : 0;
    if (fits == 0) return RRA_ERR_NOT_CORESIDENT;
    const size_t n = (size_t)c->nranks;
    const size_t ve = rra::kVecBytes / elem_size(dtype);
    memset(p, 0, sizeof(*p));
    p->win0 = c->win0;
    p->ctrl = c->ctrl;
    p->timing = c->timing;
    p->stride = c->lay.window_stride;
    p->count = count;
    p->nvec = (uint32_t)ceil_div(count, ve);
    p->timeout_ns = (uint64_t)c->timeout_ms * 1000000ull;
    p->nranks = c->nranks;
    p->nsteps = 1;
    p->chunk_vecs = p->nvec;
    p->epoch_slots = rra::kEpochSlots;
    p->root = root;
    // the bulk-copy Reduce up to 16 ranks splits each slice into N partitions,
    // as the split forms do (above 16 ranks it sends whole slices to the root)
    const bool many = c->nranks > rra::kClusterMaxRanks;
    const bool bulk_reduce = bulk && op == rra::kCollReduce && !many;
    // above 16 ranks the bulk-copy Reduce splits a slice into 16 partitions
    const bool multi_reduce = bulk && op == rra::kCollReduce && many;
    const bool split = op == rra::kCollBroadcastSplit || op == rra::kCollReduceSplit || bulk_reduce;
    // above 16 ranks a CTA hosts up to `hosted` ranks (16-CTA clusters)
    const size_t cdim = std::min<size_t>(n, rra::kClusterMaxRanks);
    const size_t hosted = ceil_div(n, cdim);
    // input vectors a CTA handles per slice position
    const size_t per_pos = (op == rra::kCollReduceScatter ? n : 1) * (op == rra::kCollBroadcast ? 1 : hosted);
    const size_t stage_vecs = rra::kClusterStageBytes / rra::kVecBytes;
    size_t smax;
    switch (op) {
        case rra::kCollBroadcast: smax = stage_vecs; break;
        case rra::kCollReduce:  // S, N S / 16 or N S vectors
            smax = bulk_reduce ? stage_vecs / n * n : multi_reduce ? (stage_vecs / n) * 16 : stage_vecs / n;
            break;
        case rra::kCollBroadcastSplit: smax = stage_vecs * n / (n + 1) / n * n; break;  // (S/N + S) vectors
        case rra::kCollReduceSplit: smax = stage_vecs / 2 / n * n; break;              // 2 S vectors
        case rra::kCollReduceScatter: smax = stage_vecs / (hosted * n); break;          // N slots per hosted owner
        default: smax = stage_vecs / n; break;
    }
    const size_t t = (size_t)c->threads;
    size_t S;
    if (c->cluster_slice > 0) {
        S = (size_t)c->cluster_slice / rra::kVecBytes;
    } else if (multi_reduce) {
        // as the bulk-copy Reduce below: about 8 clusters per SM's worth of
        // slices, at least 512 bytes per partition
        const size_t target = std::max<size_t>(1, 8 * (size_t)c->sm_count / cdim);
        S = std::max<size_t>(32 * 16, ceil_div(p->nvec, target));
    } else if (!many && (store_bulk || (bulk && (op == rra::kCollReduceScatter || op == rra::kCollReduce)))) {
        // Outputs (AllGather, Broadcast) or inputs (ReduceScatter, Reduce)
        // moved by bulk copies: the threads no longer move that data, so
        // their count does not bound the slice.  Slices for about 8 clusters
        // per SM's worth of CTAs, each window of N slots of S vectors
        // (AllGather, ReduceScatter) at most 32 KiB and at least 512 bytes per
        // slot, each Broadcast slice 4-32 KiB, each Reduce slice (N
        // partitions) at most 32 KiB and at least 512 bytes per partition.
        // (Sweeps at N = 2, 4, 8, 16 and 1-64 MiB blocks put the best slice
        // there.)
        const size_t target = std::max<size_t>(1, 8 * (size_t)c->sm_count / cdim);
        if (op == rra::kCollAllGather || op == rra::kCollReduceScatter) {
            const size_t window = std::max<size_t>(1, (32u << 10) / rra::kVecBytes / n);
            S = std::min<size_t>(window, std::max<size_t>(32, ceil_div(p->nvec, target)));
        } else if (op == rra::kCollReduce) {  // N partitions of S / N vectors, S at most 32 KiB
            S = std::min<size_t>(2048, std::max<size_t>(32 * n, ceil_div(p->nvec, target)));
            S = std::min<size_t>(S, align_up(p->nvec, n));
        } else {
            S = std::min<size_t>(2048, std::max<size_t>(256, ceil_div(p->nvec, target)));
        }
        S = std::max<size_t>(1, std::min<size_t>(S, p->nvec));
    } else {
        const size_t target = std::max<size_t>(1, 2 * (size_t)c->sm_count / cdim);
        S = std::max<size_t>(std::min<size_t>(p->nvec, std::max<size_t>(1, t / per_pos)), ceil_div(p->nvec, target));
        S = std::min<size_t>(S, std::max<size_t>(1, t * rra::kClusterBatch / per_pos));
    }
    if (split) S = align_up(S, n);  // N parts per slice
    if (multi_reduce) S = align_up(S, 16);  // 16 partitions per slice
    S = std::max<size_t>(split ? n : multi_reduce ? 16 : 1, std::min(S, smax));
    p->per_cta = (uint32_t)S;
    p->ctas_per_rank = (int32_t)ceil_div(p->nvec, S);
    *threads = (int)std::min<size_t>(t, std::max<size_t>(32, align_up(S * per_pos, 32)));
    return RRA_OK;
}

static int kernel_kind(const rra_comm* c, rra_algo_t algo) {
    const bool wide = c->oneshot_wide == 1 || (c->oneshot_wide < 0 && c->nranks >= 16);
    if (wide && (algo == RRA_ONESHOT_LL || algo == RRA_ONESHOT_SENTINEL))
        return algo == RRA_ONESHOT_LL ? rra::kKindOneshotLLWide : rra::kKindOneshotSentinelWide;
    if (wide && algo == RRA_LL128_ATOMIC) return rra::kKindLL128Wide;
    return (int)algo;
}

static rra_status_t max_ctas_kind(rra_comm* c, rra_dtype_t d, int kind, int* ctas) {
    int b = 0;
    rra_status_t st = query_blocks(c, d, kind, &b);
    if (st != RRA_OK) return st;
    *ctas = std::min(b * c->sm_count, rra::kEpochSlots);
    return RRA_OK;
}

rra_status_t rra_comm_max_coresident(rra_comm_t c, rra_dtype_t d, rra_algo_t a, int* ctas) {
    if (c == nullptr || ctas == nullptr || !valid_dtype(d) || !valid_algo(a) || a == RRA_AUTO || is_cluster(a))
        return RRA_ERR_INVALID_ARG;
    return max_ctas_kind(c, d, kernel_kind(c, a), ctas);
}

// Fills everything in Params except the pointer tables.
static rra_status_t plan_call(rra_comm* c, size_t count, rra_dtype_t dtype, rra_algo_t algo,
                              Params* p, int* kind_out, int* threads_out) {
    const size_t es = elem_size(dtype);
    const size_t ve = rra::kVecBytes / es;
    const size_t n = (size_t)c->nranks;
    const rra_layout_t& L = c->lay;
    const int kind = kernel_kind(c, algo);
    int max_ctas = 0;
    rra_status_t st = max_ctas_kind(c, dtype, kind, &max_ctas);
    if (st != RRA_OK) return st;
    *kind_out = kind;
    const int64_t cmax = std::max<int64_t>(1, max_ctas / c->nranks);
    const size_t T = (size_t)std::min(c->threads, kind_max_threads(kind));

    memset(p, 0, sizeof(*p));
    p->win0 = c->win0;
    p->ctrl = c->ctrl;
    p->timing = c->timing;
    p->trace = c->trace;
    p->stride = L.window_stride;
    p->count = count;
    p->nvec = (uint32_t)ceil_div(count, ve);
    p->timeout_ns = (uint64_t)c->timeout_ms * 1000000ull;
    p->nranks = c->nranks;
    p->epoch_slots = rra::kEpochSlots;

    // Window regions, in order (must match launch_init):
    // LL slots | barrier flags | sentinel slots | two-shot | LL128 | barrier data
    const size_t off_ll = 0;
    const size_t off_bf = off_ll + L.ll_bytes;
    const size_t off_os = off_bf + L.bf_bytes;
    const size_t off_ts = off_os + L.os_bytes;
    const size_t off_la = off_ts + L.ts_bytes;
    const size_t off_bd = off_la + L.la_bytes;
    {
        // flag regions zeroed by the epoch scrub whatever the algorithm:
        // LL slots + barrier flags (contiguous), LL128 AllGather slots
        const LaSizes ls = la_sizes(L.la_part, c->nranks);
        p->ll_off = off_ll;
        p->ll_bytes = L.ll_bytes + L.bf_bytes;
        p->llag_off = off_la + 2 * ls.acc_parity + 2 * ls.cnt_parity;
        p->llag_bytes = 2 * n * ls.ag_slot;
    }
    size_t work = 0;  // positions per step that the CTAs of one rank split
    int64_t ctas;
    switch (algo) {
        case RRA_ONESHOT_LL:
        case RRA_ONESHOT_SENTINEL: {
            const bool ll = algo == RRA_ONESHOT_LL;
            size_t cap = (ll ? L.ll_chunk : L.os_chunk) / rra::kVecBytes;
            if (c->os_chunk > 0) cap = std::min(cap, std::max<size_t>(1, (size_t)c->os_chunk / rra::kVecBytes));
            const size_t chunk = std::min<size_t>(p->nvec, cap);
            p->chunk_vecs = (uint32_t)chunk;
            p->nsteps = (uint32_t)ceil_div(p->nvec, chunk);
            p->region_off = ll ? off_ll : off_os;
            p->slot_bytes = ll ? 2 * L.ll_chunk : L.os_chunk;
            p->parity_bytes = n * p->slot_bytes;
            work = chunk;
            break;
        }
        case RRA_TWOSHOT_DBUF:
        case RRA_TWOSHOT_DIRECT: {
            size_t cap = L.ts_part / rra::kVecBytes;
            if (c->ts_chunk > 0) {
                cap = std::min(cap, std::max<size_t>(1, (size_t)c->ts_chunk / rra::kVecBytes / n));
            } else {
                // live RS (+AG) scratch: N windows x 2 parities x N slots x part
                cap = std::min(cap, std::max<size_t>(64, kLiveScratch / (2 * n * n) / rra::kVecBytes));
                // one position per thread per step on the largest co-resident
                // grid (GB300 sweep at N = 8, 16-64 MiB per rank: 2.1x the
                // bandwidth of 1.7 positions per thread in 2 MiB steps)
                cap = std::min(cap, (size_t)cmax * T);
            }
            const size_t part = std::min(ceil_div(p->nvec, n), cap);
            p->chunk_vecs = (uint32_t)part;
            p->nsteps = (uint32_t)ceil_div(p->nvec, n * part);
            p->region_off = off_ts;
            p->slot_bytes = L.ts_part;
            p->parity_bytes = n * L.ts_part;
            p->aux_off = off_ts + 2 * p->parity_bytes;
            work = part;
            break;
        }
        case RRA_LL128_ATOMIC: {
            size_t cap = L.la_part / rra::kVecBytes;
            if (c->la_chunk > 0)
                cap = std::min(cap, std::max<size_t>(1, (size_t)c->la_chunk / rra::kVecBytes / n));
            else  // live accumulators + LL AllGather slots: about 4 N^2 x part
                cap = std::min(cap, std::max<size_t>(64, kLiveScratchLL128 / (4 * n * n) / rra::kVecBytes));
            const size_t part = std::min(ceil_div(p->nvec, n), cap);
            const LaSizes s = la_sizes(L.la_part, c->nranks);
            p->chunk_vecs = (uint32_t)part;
            p->nsteps = (uint32_t)ceil_div(p->nvec, n * part);
            p->region_off = off_la;
            p->parity_bytes = s.acc_parity;
            p->aux_off = off_la + 2 * s.acc_parity;
            p->aux_parity_bytes = s.cnt_parity;
            p->aux2_off = p->aux_off + 2 * s.cnt_parity;
            p->aux2_slot_bytes = s.ag_slot;
            p->aux2_parity_bytes = n * s.ag_slot;
            work = part;
            break;
        }
        case RRA_ONESHOT_BARRIER: {
            size_t cap = L.bd_chunk / rra::kVecBytes;
            if (c->os_chunk > 0) cap = std::min(cap, std::max<size_t>(1, (size_t)c->os_chunk / rra::kVecBytes));
            const size_t chunk = std::min<size_t>(p->nvec, cap);
            p->chunk_vecs = (uint32_t)chunk;
            p->nsteps = (uint32_t)ceil_div(p->nvec, chunk);
            p->region_off = off_bd;
            p->slot_bytes = L.bd_chunk;
            p->parity_bytes = 0;
            p->aux_off = off_bf;
            work = chunk;
            break;
        }
        case RRA_TWOSHOT_BARRIER: {
            // partitions of at most one slot (bd_chunk); a step covers N of them
            size_t part = L.bd_chunk / rra::kVecBytes;
            if (c->ts_chunk > 0) part = std::min(part, std::max<size_t>(1, (size_t)c->ts_chunk / rra::kVecBytes / n));
            part = std::min(part, ceil_div(p->nvec, n));
            p->chunk_vecs = (uint32_t)(n * part);
            p->nsteps = (uint32_t)ceil_div(p->nvec, n * part);
            p->region_off = off_bd;                      // ReduceScatter slots [q]
            p->aux2_off = off_bd + n * L.bd_chunk;       // AllGather slots [q]
            p->slot_bytes = L.bd_chunk;
            p->parity_bytes = 0;
            p->aux_off = off_bf;
            work = part;
            break;
        }
        default:
            return RRA_ERR_INVALID_ARG;
    }
    int64_t cap_ctas = cmax;
    if (algo == RRA_ONESHOT_BARRIER || algo == RRA_TWOSHOT_BARRIER)
        cap_ctas = std::min<int64_t>(cap_ctas, rra::kBarrierCtas);
    const bool wide = kind == rra::kKindOneshotLLWide || kind == rra::kKindOneshotSentinelWide;
    const bool wide_la = kind == rra::kKindLL128Wide;
    // positions per CTA to aim for: one per thread; for the wide one-shot, as
    // many as one shared-memory stage round holds; for the wide LL128-atomic,
    // about 8 (owner, position) items per thread
    const size_t target = wide ? std::max<size_t>(32, (size_t)rra::kWideStageVecs / n)
                               : wide_la ? std::max<size_t>(32, 8 * T / n) : T;
    if (c->ctas_per_rank > 0) ctas = std::min<int64_t>(c->ctas_per_rank, cap_ctas);
    else ctas = std::min<int64_t>((int64_t)ceil_div(work, target), cap_ctas);
    ctas = std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)work));
    size_t per = ceil_div(work, (size_t)ctas);
    if (algo == RRA_LL128_ATOMIC) per = align_up(per, rra::kGroupVecs);
    ctas = (int64_t)ceil_div(work, per);
    p->ctas_per_rank = (int32_t)ctas;
    p->per_cta = (uint32_t)per;
    // Small CTAs for small per-CTA work (fewer idle warps to launch and
    // retire); never below 64 threads (the barrier baseline needs one thread
    // per rank), never above the occupancy-checked size.
    int threads = (int)T;
    if (wide_la) threads = (int)std::min<size_t>(T, std::max<size_t>(64, align_up(n * std::min(per, work), 32)));
    else if (!wide) threads = (int)std::min<size_t>(T, std::max<size_t>(64, align_up(per, 32)));
    *threads_out = threads;
    return RRA_OK;
}

rra_status_t rra_comm_plan_call(rra_comm_t c, size_t count, rra_dtype_t dtype, rra_algo_t algo,
                                int* grid_ctas, int* steps) {
    if (c == nullptr || !valid_dtype(dtype) || !valid_algo(algo) || count == 0) return RRA_ERR_INVALID_ARG;
    if (count > c->max_bytes / elem_size(dtype)) return RRA_ERR_INVALID_ARG;
    const bool autoselect = algo == RRA_AUTO;
    if (autoselect) algo = select_cluster(c->nranks, count * elem_size(dtype), c->cluster_tma != 0);
    Params p;
    int kind = 0, threads = 0;
    rra_status_t st = is_cluster(algo) ? plan_cluster(c, count, dtype, algo, &p, &threads, &kind, false, true)
                                       : plan_call(c, count, dtype, algo, &p, &kind, &threads);
    if (st == RRA_ERR_NOT_CORESIDENT && autoselect && is_cluster(algo)) {
        algo = select_global(c->nranks, count * elem_size(dtype));
        st = plan_call(c, count, dtype, algo, &p, &kind, &threads);
    }
    if (st != RRA_OK) return st;
    const bool multi = is_cluster(algo) && (kind == rra::kClusterOneshotMulti || kind == rra::kClusterTwoshotMulti);
    if (grid_ctas) *grid_ctas = (multi ? rra::kClusterMaxRanks : p.nranks) * p.ctas_per_rank;
    if (steps) *steps = (int)p.nsteps;
    return RRA_OK;
}

static const char* kernel_name(bool cluster, int kind) {
    if (cluster) {
        switch (kind) {
            case rra::kClusterOneshot: return "cluster_kernel<one-shot>";
            case rra::kClusterTwoshot: return "cluster_kernel<two-shot>";
            case rra::kClusterTwoshotPipe: return "cluster_pipe_kernel";
            case rra::kClusterOneshotMulti: return "cluster_multi_kernel<one-shot>";
            case rra::kClusterTwoshotMulti: return "cluster_multi_kernel<two-shot>";
            case rra::kClusterOneshotMultiTma: return "cluster_multi_kernel<one-shot, bulk>";
            case rra::kClusterTwoshotMultiTma: return "cluster_multi_kernel<two-shot, bulk>";
            case rra::kClusterOneshotTma: return "cluster_tma_kernel<one-shot>";
            case rra::kClusterTwoshotTma: return "cluster_tma_kernel<two-shot>";
        }
        return "unknown";
    }
    switch (kind) {
        case rra::kKindOneshotLL: return "oneshot_kernel<LL>";
        case rra::kKindOneshotSentinel: return "oneshot_kernel<sentinel>";
        case rra::kKindTwoshot: return "twoshot_kernel<scratch>";
        case rra::kKindTwoshotDirect: return "twoshot_kernel<direct>";
        case rra::kKindLL128: return "ll128_kernel";
        case rra::kKindLL128Wide: return "ll128_wide_kernel";
        case rra::kKindOneshotLLWide: return "oneshot_wide_kernel<LL>";
        case rra::kKindOneshotSentinelWide: return "oneshot_wide_kernel<sentinel>";
        case rra::kKindOneshotBarrier: return "oneshot_barrier_kernel";
        case rra::kKindTwoshotBarrier: return "twoshot_barrier_kernel";
    }
    return "unknown";
}

// The plan of a call on device buffers of this GPU (bulk-copy push allowed).
rra_status_t rra_comm_plan_kernel(rra_comm_t c, size_t count, rra_dtype_t dtype, rra_algo_t algo,
                                  const char** name) {
    if (c == nullptr || name == nullptr || !valid_dtype(dtype) || !valid_algo(algo) || count == 0)
        return RRA_ERR_INVALID_ARG;
    if (count > c->max_bytes / elem_size(dtype)) return RRA_ERR_INVALID_ARG;
    const bool autoselect = algo == RRA_AUTO;
    if (autoselect) algo = select_cluster(c->nranks, count * elem_size(dtype), c->cluster_tma != 0);
    Params p;
    int kind = 0, threads = 0;
    std::lock_guard<std::mutex> g(c->mu);
    rra_status_t st = is_cluster(algo) ? plan_cluster(c, count, dtype, algo, &p, &threads, &kind, false, true)
                                       : plan_call(c, count, dtype, algo, &p, &kind, &threads);
    if (st == RRA_ERR_NOT_CORESIDENT && autoselect && is_cluster(algo)) {
        algo = select_global(c->nranks, count * elem_size(dtype));
        st = plan_call(c, count, dtype, algo, &p, &kind, &threads);
    }
    if (st != RRA_OK) return st;
    *name = kernel_name(is_cluster(algo), kind);
    return RRA_OK;
}

static rra_status_t run_allreduce(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                                  rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream, bool host);

rra_status_t rra_allreduce(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                           rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream) {
    return run_allreduce(c, send, recv, count, dtype, algo, stream, false);
}

static rra_status_t run_allreduce(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                                  rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream, bool host) {
    if (c == nullptr || send == nullptr || recv == nullptr) return RRA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_algo(algo)) return RRA_ERR_INVALID_ARG;
    if (c->poisoned) return RRA_ERR_POISONED;
    if (count == 0) return RRA_OK;
    const size_t es = elem_size(dtype);
    if (count > c->max_bytes / es) return RRA_ERR_INVALID_ARG;
    const bool autoselect = algo == RRA_AUTO;
    Params p;
    int kind = 0, threads = 0;
    {
        std::lock_guard<std::mutex> g(c->mu);
        // bulk copies only from this GPU's own device memory (never host buffers)
        const bool local = !host && bulk_copy_push(c) && bulk_sources_local(c, send, c->nranks, count * es);
        if (autoselect) algo = select_cluster(c->nranks, count * es, local);
        rra_status_t st = is_cluster(algo) ? plan_cluster(c, count, dtype, algo, &p, &threads, &kind, host, local)
                                           : plan_call(c, count, dtype, algo, &p, &kind, &threads);
        if (st == RRA_ERR_NOT_CORESIDENT && autoselect && is_cluster(algo)) {
            algo = select_global(c->nranks, count * es);
            st = plan_call(c, count, dtype, algo, &p, &kind, &threads);
        }
        if (st != RRA_OK) return st;
        c->last_kernel = kernel_name(is_cluster(algo), kind);
    }
    for (int r = 0; r < c->nranks; ++r) {
        if (send[r] == nullptr || recv[r] == nullptr) return RRA_ERR_INVALID_ARG;
        if (((uintptr_t)send[r] | (uintptr_t)recv[r]) & 15u) return RRA_ERR_INVALID_ARG;
        p.send[r] = send[r];
        p.recv[r] = recv[r];
    }
    p.drop_rank = c->drop_rank;
    cudaError_t e = is_cluster(algo)
                        ? rra::launch_cluster(p, dtype, kind, threads, (cudaStream_t)stream, c->pdl != 0)
                        : rra::launch_allreduce(p, dtype, kind, threads, (cudaStream_t)stream, c->cooperative != 0,
                                                c->pdl != 0);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return RRA_ERR_NOT_CORESIDENT;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    return RRA_OK;
}

// After `s` completes: the status of the calls on it, from the
// device-written host mirror (or by copying the status word back).
static rra_status_t sync_status(rra_comm* c, cudaStream_t s) {
    if (!c->host_mirror &&
        cudaMemcpyAsync(c->host_status, &c->ctrl->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
        return RRA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RRA_ERR_CUDA;
    const uint32_t v = *(volatile uint32_t*)c->host_status;
    if (v != 0u) {
        c->poisoned = true;
        return (rra_status_t)v;
    }
    return RRA_OK;
}

rra_status_t rra_host_device_ptrs(int n, const void* const host[], void* dev[]) {
    if (n < 0 || n > 2 * RRA_MAX_RANKS || (n > 0 && (host == nullptr || dev == nullptr))) return RRA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        dev[i] = nullptr;
        if (host[i] == nullptr) continue;
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, host[i]) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) dev[i] = a.devicePointer;
    }
    return RRA_OK;
}

rra_status_t rra_allreduce_mapped(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                                  rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    if (c->host_status == nullptr) return RRA_ERR_OOM;  // its allocation failed at creation
    rra_status_t st = run_allreduce(c, send, recv, count, dtype, algo, stream, true);
    if (st != RRA_OK || count == 0) return st;
    return sync_status(c, (cudaStream_t)stream);
}

rra_status_t rra_allreduce_host(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                                rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream) {
    if (c == nullptr || send == nullptr || recv == nullptr) return RRA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_algo(algo)) return RRA_ERR_INVALID_ARG;
    if (c->poisoned) return RRA_ERR_POISONED;
    if (count == 0) return RRA_OK;
    const size_t es = elem_size(dtype);
    if (count > c->max_bytes / es) return RRA_ERR_INVALID_ARG;
    for (int r = 0; r < c->nranks; ++r)
        if (send[r] == nullptr || recv[r] == nullptr) return RRA_ERR_INVALID_ARG;
    if (c->host_status == nullptr) return RRA_ERR_OOM;  // its allocation failed at creation
    cudaStream_t s = (cudaStream_t)stream;
    auto finish = [&]() -> rra_status_t { return sync_status(c, s); };
    // Zero copy: when every buffer is pinned host memory that the device can
    // address (on GB300, reached over the coherent NVLink-C2C link to the
    // Grace CPU), the kernel reads the inputs and writes the outputs in host
    // memory itself; no staging buffers and no copies.
    if (c->host_zero_copy) {
        const void* msend[RRA_MAX_RANKS];
        void* mrecv[RRA_MAX_RANKS];
        bool mapped = true;
        for (int r = 0; r < c->nranks && mapped; ++r) {
            cudaPointerAttributes a{}, b{};
            if (cudaPointerGetAttributes(&a, send[r]) != cudaSuccess ||
                cudaPointerGetAttributes(&b, recv[r]) != cudaSuccess || a.type != cudaMemoryTypeHost ||
                b.type != cudaMemoryTypeHost || a.devicePointer == nullptr || b.devicePointer == nullptr) {
                cudaGetLastError();
                mapped = false;
                break;
            }
            msend[r] = a.devicePointer;
            mrecv[r] = b.devicePointer;
        }
        if (mapped) {
            rra_status_t st = run_allreduce(c, msend, mrecv, count, dtype, algo, stream, true);
            if (st != RRA_OK) return st;
            return finish();
        }
    }
    if (c->stage == nullptr) {
        c->stage_slot = align_up(c->max_bytes, 256);
        if (cudaMalloc((void**)&c->stage, 2 * (size_t)c->nranks * c->stage_slot) != cudaSuccess) {
            cudaGetLastError();
            c->stage = nullptr;
            return RRA_ERR_OOM;
        }
    }
    const size_t bytes = count * es;
    const void* dsend[RRA_MAX_RANKS];
    void* drecv[RRA_MAX_RANKS];
    for (int r = 0; r < c->nranks; ++r) {
        dsend[r] = c->stage + (size_t)r * c->stage_slot;
        drecv[r] = c->stage + (size_t)(c->nranks + r) * c->stage_slot;
        if (cudaMemcpyAsync((void*)dsend[r], send[r], bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return RRA_ERR_CUDA;
    }
    rra_status_t st = rra_allreduce(c, dsend, drecv, count, dtype, algo, stream);
    if (st != RRA_OK) return st;
    for (int r = 0; r < c->nranks; ++r) {
        if (cudaMemcpyAsync(recv[r], drecv[r], bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return RRA_ERR_CUDA;
    }
    return finish();
}

// Shared front end of the four collectives.  ReduceScatter's inputs and
// AllGather's outputs hold nranks blocks of `count` elements; those must fit
// max_bytes.  Broadcast reads only send[root]; Reduce writes only recv[root].
static rra_status_t run_coll(rra_comm_t c, int op, int root, const void* const send[], void* const recv[],
                             size_t count, rra_dtype_t dtype, rra_stream_t stream) {
    if (c == nullptr || send == nullptr || recv == nullptr || !valid_dtype(dtype)) return RRA_ERR_INVALID_ARG;
    if ((op == rra::kCollBroadcast || op == rra::kCollReduce) && (root < 0 || root >= c->nranks))
        return RRA_ERR_INVALID_ARG;
    if (c->poisoned) return RRA_ERR_POISONED;
    if (count == 0) return RRA_OK;
    const size_t es = elem_size(dtype);
    const size_t blocks = (op == rra::kCollReduceScatter || op == rra::kCollAllGather) ? (size_t)c->nranks : 1;
    if (count > c->max_bytes / es / blocks) return RRA_ERR_INVALID_ARG;
    Params p;
    int threads = 0;
    bool bulk = false, store_bulk = false;
    {
        std::lock_guard<std::mutex> g(c->mu);
        // AllGather and Broadcast (up to 16 ranks) push by bulk copies from
        // the senders' inputs, when those are device memory of this GPU; and
        // write their outputs by bulk copies too, when those are device
        // memory of this GPU and a block is whole 16-byte vectors, from 4 KiB
        // blocks (AllGather) or 256 KiB (Broadcast) up: below, the vector
        // stores measured faster
        // ReduceScatter pushes by bulk copies as well (one per owner) when a
        // block is whole 16-byte vectors, so that every block starts aligned.
        const bool rs = op == rra::kCollReduceScatter;
        if (rra::coll_has_bulk(op, c->nranks) && c->cluster_tma != 0 && (!rs || (count * es) % rra::kVecBytes == 0)) {
            const int nsrc = op == rra::kCollBroadcast ? 1 : c->nranks;
            const void* const* src = op == rra::kCollBroadcast ? send + root : send;
            bulk = bulk_sources_local(c, src, nsrc, (rs ? (size_t)c->nranks : 1u) * count * es);
            const size_t store_min = op == rra::kCollBroadcast ? (256u << 10) : (4u << 10);
            const bool may_store = op == rra::kCollAllGather || op == rra::kCollBroadcast;
            if (bulk && may_store && (count * es) % rra::kVecBytes == 0 && count * es >= store_min) {
                const void* out[RRA_MAX_RANKS];
                for (int r = 0; r < c->nranks; ++r) out[r] = recv[r];
                store_bulk = bulk_sources_local(c, out, c->nranks, blocks * count * es);
            }
        }
        // Broadcast / Reduce: two hops for large messages (the root's CTA no
        // longer carries all of a slice's traffic), one hop for small ones --
        // except a Broadcast whose copies are all bulk copies, which stays one
        // hop (the root's slice reaches every CTA in one multicast copy); the
        // two-hop forms exist for up to 16 ranks
        if ((op == rra::kCollBroadcast || op == rra::kCollReduce) && c->nranks <= rra::kClusterMaxRanks) {
            // (the bulk-copy Reduce is already spread over the cluster)
            const bool one_hop_bulk = store_bulk || (bulk && op == rra::kCollReduce);
            const bool split = c->coll_split == 1 ||
                               (c->coll_split < 0 && !one_hop_bulk && c->nranks >= 3 && count * es >= (256u << 10));
            if (split) {
                op = op == rra::kCollBroadcast ? rra::kCollBroadcastSplit : rra::kCollReduceSplit;
                bulk = store_bulk = false;
            }
        }
        rra_status_t st = plan_coll(c, count, dtype, op, root < 0 ? 0 : root, bulk, store_bulk, &p, &threads);
        if (st != RRA_OK) return st;
        c->last_kernel = rra::coll_kernel_name(op, c->nranks, bulk, store_bulk);
    }
    const bool bcast = op == rra::kCollBroadcast || op == rra::kCollBroadcastSplit;
    const bool reduce = op == rra::kCollReduce || op == rra::kCollReduceSplit;
    for (int r = 0; r < c->nranks; ++r) {
        const bool need_send = !bcast || r == root;  // Broadcast reads only the root's input
        const bool need_recv = !reduce || r == root;  // Reduce writes only the root's output
        if ((need_send && send[r] == nullptr) || (need_recv && recv[r] == nullptr)) return RRA_ERR_INVALID_ARG;
        if (((uintptr_t)(need_send ? send[r] : nullptr) | (uintptr_t)(need_recv ? recv[r] : nullptr)) & 15u)
            return RRA_ERR_INVALID_ARG;
        p.send[r] = need_send ? send[r] : nullptr;
        p.recv[r] = need_recv ? recv[r] : nullptr;
    }
    p.drop_rank = c->drop_rank;
    cudaError_t e = rra::launch_coll(p, dtype, op, threads, (cudaStream_t)stream, c->pdl != 0, bulk, store_bulk);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    return RRA_OK;
}

rra_status_t rra_reduce_scatter(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                                rra_dtype_t dtype, rra_stream_t stream) {
    return run_coll(c, rra::kCollReduceScatter, -1, send, recv, count, dtype, stream);
}

rra_status_t rra_all_gather(rra_comm_t c, const void* const send[], void* const recv[], size_t count,
                            rra_dtype_t dtype, rra_stream_t stream) {
    return run_coll(c, rra::kCollAllGather, -1, send, recv, count, dtype, stream);
}

rra_status_t rra_broadcast(rra_comm_t c, int root, const void* const send[], void* const recv[], size_t count,
                           rra_dtype_t dtype, rra_stream_t stream) {
    return run_coll(c, rra::kCollBroadcast, root, send, recv, count, dtype, stream);
}

rra_status_t rra_reduce(rra_comm_t c, int root, const void* const send[], void* const recv[], size_t count,
                        rra_dtype_t dtype, rra_stream_t stream) {
    return run_coll(c, rra::kCollReduce, root, send, recv, count, dtype, stream);
}

// AllReduce + residual add (fused.cu): the shape (one- or two-shot) and the
// push (bulk copies or st.async) that RRA_AUTO's cluster AllReduce would
// take.  Slices as for the cluster AllReduce, within a stage of two
// sub-buffers; one cluster per slice unless RRA_ATTR_CTAS_PER_RANK caps the
// clusters (then each loops over several slices, one epoch each).
// local: every send[r] is device memory of this GPU (bulk_sources_local).
static rra_status_t plan_residual(rra_comm* c, size_t count, rra_dtype_t dtype, rra::FusedParams* f,
                                  int* threads, bool* two_shot, bool* bulk_out, bool local) {
    *bulk_out = false;
    const size_t n = (size_t)c->nranks;
    const size_t es = elem_size(dtype);
    if (c->nranks > rra::kClusterMaxRanks) {
        // the many-rank cluster AllReduce's plan and shape choice (RRA_AUTO's
        // 16 N M <= 1 MiB), with the residual add in the kernel's epilogue
        const bool two = (size_t)rra::kClusterMaxRanks * n * count * es > (1ull << 20);
        const int rmode = two ? rra::kClusterTwoshotMultiRes : rra::kClusterOneshotMultiRes;
        int& fits = c->residual_multi_fits[two ? 1 : 0][(int)dtype];
        if (fits < 0)
            fits = rra::cluster_max_active(dtype, rmode, c->nranks, 256, rra::kClusterStageBytes) > 0 ? 1 : 0;
        if (fits == 0) return RRA_ERR_NOT_CORESIDENT;
        memset(f, 0, sizeof(*f));
        int mode = 0;
        rra_status_t st = plan_cluster_multi(c, count, dtype, two, &f->base, threads, &mode, false);
        if (st != RRA_OK) return st;
        *two_shot = two;
        return RRA_OK;
    }
    // shape and push as the cluster AllReduce would take them
    const bool bulk = bulk_copy_push(c) && local && c->nranks <= rra::kClusterMaxRanks;
    const bool two = select_cluster(c->nranks, count * es, bulk) == RRA_TWOSHOT_CLUSTER;
    int& fits = c->residual_fits[bulk ? 1 : 0][two ? 1 : 0][(int)dtype];
    if (fits < 0)
        fits = rra::residual_max_active(dtype, two, bulk, c->nranks, 256, rra::kClusterStageBytes) > 0 ? 1 : 0;
    if (fits == 0) return RRA_ERR_NOT_CORESIDENT;
    memset(f, 0, sizeof(*f));
    rra::Params* p = &f->base;
    p->win0 = c->win0;
    p->ctrl = c->ctrl;
    p->timing = c->timing;
    p->trace = c->trace;
    p->stride = c->lay.window_stride;
    p->count = count;
    p->nvec = (uint32_t)ceil_div(count, rra::kVecBytes / es);
    p->timeout_ns = (uint64_t)c->timeout_ms * 1000000ull;
    p->nranks = c->nranks;
    p->chunk_vecs = p->nvec;
    p->epoch_slots = rra::kEpochSlots;
    const size_t half = rra::kClusterStageBytes / 2 / rra::kVecBytes;  // vectors per sub-buffer
    const size_t smax = two ? half / n * n : half / n;
    const size_t t = (size_t)c->threads;
    size_t S;
    if (c->cluster_slice > 0) {
        S = (size_t)c->cluster_slice / rra::kVecBytes;
    } else {
        const size_t target = std::max<size_t>(1, 2 * (size_t)c->sm_count / n);
        S = std::max<size_t>(std::min<size_t>(p->nvec, t), ceil_div(p->nvec, target));
        S = std::min<size_t>(S, t * rra::kClusterBatch);
    }
    if (two) S = align_up(S, n);
    S = std::max<size_t>(two ? n : 1, std::min(S, smax));
    const size_t nslices = ceil_div(p->nvec, S);
    p->per_cta = (uint32_t)S;
    p->nsteps = (uint32_t)nslices;
    p->ctas_per_rank = (int32_t)(c->ctas_per_rank > 0 ? std::min(nslices, (size_t)c->ctas_per_rank) : nslices);
    *threads = (int)std::min<size_t>(t, std::max<size_t>(32, align_up(S, 32)));
    *two_shot = two;
    *bulk_out = bulk;
    return RRA_OK;
}

rra_status_t rra_allreduce_residual(rra_comm_t c, const void* const send[], const void* const residual[],
                                    void* const recv[], size_t count, rra_dtype_t dtype, rra_stream_t stream) {
    if (c == nullptr || send == nullptr || residual == nullptr || recv == nullptr || !valid_dtype(dtype))
        return RRA_ERR_INVALID_ARG;
    if (c->poisoned) return RRA_ERR_POISONED;
    if (count == 0) return RRA_OK;
    if (count > c->max_bytes / elem_size(dtype)) return RRA_ERR_INVALID_ARG;
    rra::FusedParams f;
    int threads = 0;
    bool two = false, bulk = false, tma_res = false;
    {
        std::lock_guard<std::mutex> g(c->mu);
        const size_t bytes = count * elem_size(dtype);
        const bool local = bulk_copy_push(c) && bulk_sources_local(c, send, c->nranks, bytes);
        // Up to 16 ranks, the one-shot shape on bulk copies with one slice per
        // cluster: the cluster AllReduce's bulk-copy one-shot, planned as for
        // rra_allreduce, with the residual add in its epilogue (N = 8, bf16
        // [B, 8192]: B = 1 in 1.1 us in the kernel, B = 4 in 1.3 us, against
        // 1.8 and 2.0 us for the device-API kernel below; at two-shot sizes
        // that kernel stays faster than the same epilogue on the cluster
        // two-shot)
        if (c->nranks <= rra::kClusterMaxRanks && local && c->ctas_per_rank <= 0 && c->cluster_pipe == 0 &&
            select_cluster(c->nranks, bytes, true) == RRA_ONESHOT_CLUSTER) {
            int mode = 0;
            rra_status_t st = plan_cluster(c, count, dtype, RRA_ONESHOT_CLUSTER, &f.base, &threads, &mode, false, true);
            if (st != RRA_OK) return st;
            tma_res = mode == rra::kClusterOneshotTma;
        }
        if (!tma_res) {
            rra_status_t st = plan_residual(c, count, dtype, &f, &threads, &two, &bulk, local);
            if (st != RRA_OK) return st;
        }
        c->last_kernel = tma_res ? "cluster_tma_kernel<one-shot, residual>"
                         : c->nranks > rra::kClusterMaxRanks
                             ? (two ? "residual_multi_kernel<two-shot>" : "residual_multi_kernel<one-shot>")
                         : bulk ? (two ? "residual_kernel<two-shot, bulk>" : "residual_kernel<one-shot, bulk>")
                                : (two ? "residual_kernel<two-shot>" : "residual_kernel<one-shot>");
    }
    for (int r = 0; r < c->nranks; ++r) {
        if (send[r] == nullptr || residual[r] == nullptr || recv[r] == nullptr) return RRA_ERR_INVALID_ARG;
        if (((uintptr_t)send[r] | (uintptr_t)residual[r] | (uintptr_t)recv[r]) & 15u) return RRA_ERR_INVALID_ARG;
        f.base.send[r] = send[r];
        f.base.recv[r] = recv[r];
        f.resid[r] = residual[r];
    }
    f.base.drop_rank = c->drop_rank;
    cudaError_t e = tma_res ? rra::launch_cluster_tma_residual(f, dtype, threads, (cudaStream_t)stream, c->pdl != 0)
                    : c->nranks > rra::kClusterMaxRanks
                        ? rra::launch_cluster_residual(f, dtype, two, threads, (cudaStream_t)stream, c->pdl != 0)
                        : rra::launch_residual(f, dtype, two, bulk, threads, (cudaStream_t)stream, c->pdl != 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_CUDA;
    }
    return RRA_OK;
}

// Synchronises, reads the status word and where it was recorded.
static rra_status_t read_status(rra_comm* c, int* rank, int* step) {
    if (cudaDeviceSynchronize() != cudaSuccess) return RRA_ERR_CUDA;
    uint32_t hdr[3];
    if (cudaMemcpy(hdr, c->ctrl, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return RRA_ERR_CUDA;
    if (rank) *rank = hdr[0] ? (int)(int32_t)hdr[1] : -1;
    if (step) *step = hdr[0] ? (int)(int32_t)hdr[2] : -1;
    if (hdr[0] != 0u) {
        c->poisoned = true;
        return (rra_status_t)hdr[0];
    }
    return c->poisoned ? RRA_ERR_POISONED : RRA_OK;
}

rra_status_t rra_comm_status(rra_comm_t c) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    return read_status(c, nullptr, nullptr);
}

rra_status_t rra_comm_error_site(rra_comm_t c, int* rank, int* step) {
    if (c == nullptr || rank == nullptr || step == nullptr) return RRA_ERR_INVALID_ARG;
    const rra_status_t st = read_status(c, rank, step);
    return st == RRA_ERR_CUDA || st == RRA_ERR_INVALID_ARG ? st : RRA_OK;
}

rra_status_t rra_comm_last_kernel(rra_comm_t c, const char** name) {
    if (c == nullptr || name == nullptr) return RRA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(c->mu);
    *name = c->last_kernel;
    return RRA_OK;
}

rra_status_t rra_comm_reset(rra_comm_t c) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return RRA_ERR_CUDA;
    if (rra::launch_init(c->base, c->lay.total_bytes, c->lay, c->nranks, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return RRA_ERR_CUDA;
    if (c->host_status) *(volatile uint32_t*)c->host_status = 0u;
    std::lock_guard<std::mutex> g(c->mu);
    c->poisoned = false;
    c->drop_rank = -1;
    c->local_sources.clear();
    return RRA_OK;
}

rra_status_t rra_comm_set_timing(rra_comm_t c, uint64_t* dev_buf) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(c->mu);
    c->timing = dev_buf;
    return RRA_OK;
}

rra_status_t rra_comm_barrier_latency(rra_comm_t c, int iters, double* ns_per_barrier) {
    if (c == nullptr || ns_per_barrier == nullptr || iters < 2 || iters > (1 << 24)) return RRA_ERR_INVALID_ARG;
    if (c->poisoned) return RRA_ERR_POISONED;
    Params p;
    int kind = 0, threads = 0;
    rra_status_t st;
    {
        std::lock_guard<std::mutex> g(c->mu);
        st = plan_call(c, 1, RRA_FP32, RRA_ONESHOT_BARRIER, &p, &kind, &threads);
    }
    if (st != RRA_OK) return st;
    uint64_t* dt = nullptr;
    if (cudaMalloc((void**)&dt, 2 * sizeof(uint64_t)) != cudaSuccess) {
        cudaGetLastError();
        return RRA_ERR_OOM;
    }
    p.ctas_per_rank = 1;
    p.per_cta = 1;
    p.nsteps = (uint32_t)iters;
    p.timing = dt;
    p.drop_rank = c->drop_rank;
    uint64_t h[2] = {0, 0};
    st = RRA_OK;
    if (rra::launch_allreduce(p, RRA_FP32, rra::kKindBarrierProbe, 128, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(h, dt, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        st = RRA_ERR_CUDA;
    }
    cudaFree(dt);
    if (st != RRA_OK) return st;
    st = read_status(c, nullptr, nullptr);
    if (st != RRA_OK) return st;
    *ns_per_barrier = (double)(h[1] - h[0]) / (double)(iters - 1);
    return RRA_OK;
}

rra_status_t rra_comm_get_epoch(rra_comm_t c, uint64_t* epoch) {
    if (c == nullptr || epoch == nullptr) return RRA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return RRA_ERR_CUDA;
    uint64_t m1 = 0;
    if (cudaMemcpy(&m1, &c->ctrl->epoch_m1[0], sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RRA_ERR_CUDA;
    *epoch = m1 + 1;
    return RRA_OK;
}

rra_status_t rra_comm_set_epoch(rra_comm_t c, uint64_t epoch) {
    if (c == nullptr || epoch == 0) return RRA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return RRA_ERR_CUDA;
    uint64_t* h = (uint64_t*)malloc(sizeof(uint64_t) * rra::kEpochSlots);
    if (h == nullptr) return RRA_ERR_OOM;
    for (int i = 0; i < rra::kEpochSlots; ++i) h[i] = epoch - 1;
    const cudaError_t e =
        cudaMemcpy(c->ctrl->epoch_m1, h, sizeof(uint64_t) * rra::kEpochSlots, cudaMemcpyHostToDevice);
    free(h);
    return e == cudaSuccess ? RRA_OK : RRA_ERR_CUDA;
}

rra_status_t rra_comm_set_trace(rra_comm_t c, uint64_t* dev_buf) {
    if (c == nullptr) return RRA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(c->mu);
    c->trace = dev_buf;
    return RRA_OK;
}

rra_status_t rra_comm_inject_drop(rra_comm_t c, int rank) {
    if (c == nullptr || rank < -1 || rank >= c->nranks) return RRA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return RRA_ERR_CUDA;
    std::lock_guard<std::mutex> g(c->mu);
    c->drop_rank = rank;
    return RRA_OK;
}

}  // extern "C"
