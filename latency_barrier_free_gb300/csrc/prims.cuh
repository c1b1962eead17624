// prims.cuh -- device primitives: memory-model-explicit loads/stores, fences,
// vector atomics, LL packing, sentinel tests and bounded waits.
//
// Memory-model notes (PTX ISA memory consistency model):
//  * Scratch written by one virtual rank and read by another is accessed only
//    with .relaxed.gpu (or stronger) operations, so the accesses are morally
//    strong, bypass the non-coherent L1, and meet at L2.
//  * A vector access is a set of element accesses; each aligned element of
//    up to 64 bits is single-copy atomic.  The LL protocol therefore puts a
//    32-bit payload and its 32-bit epoch flag in ONE 64-bit element.
//  * fence.acq_rel.gpu after relaxed polls and before relaxed stores gives
//    the acquire/release pairs that make "receive grants credit for the next
//    send" ("Every Microsecond Matters", Sec. IV, double buffering) hold.
#pragma once

#include <stdint.h>

#include <cuda_bf16.h>

#include "rra_internal.h"

namespace rra {

// ---------------------------------------------------------------- loads ----
// Input vector: read-only path, no L1 allocation (each byte is read once).
__device__ __forceinline__ uint4 ld_input_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void ld_relaxed_v2u64(const void* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];"
                 : "=l"(a), "=l"(b)
                 : "l"(p)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const void* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// --------------------------------------------------------------- stores ----
__device__ __forceinline__ void st_relaxed_v4(void* p, uint4 v) {
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_relaxed_v2u64(void* p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" : : "l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(void* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(void* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" : : "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_weak_u64(void* p, uint64_t v) {
    asm volatile("st.global.u64 [%0], %1;" : : "l"(p), "l"(v) : "memory");
}

// Output vector: plain store.
__device__ __forceinline__ void st_output_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// L2 prefetch of one line: also brings the address translation into the SM,
// so a later store/poll to that page does not wait for it.
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" : : "l"(p));
}

// ------------------------------------------- programmatic dependent launch ----
// A kernel waits for its predecessor (griddepcontrol.wait) before it touches
// global memory, and releases its successor (griddepcontrol.launch_dependents)
// so that the next launch overlaps it.  Where: a grid of one cluster (or one
// CTA) releases at entry -- it holds a few SMs, so successors launched ahead
// cost little, and the early release hides the next launch; a larger grid
// releases only once it is past its own wait, so a chain of calls runs at
// most one kernel ahead.  (Released at entry, a CUDA graph of 160 calls at
// N = 8, bf16 [4, 8192] launched several kernels ahead, whose waiting CTAs
// held SMs: 2.58 us per call against 1.59 us; released after the wait, a
// one-cluster call at N = 4, 128 B took one or two 128 ns steps longer.)
__device__ __forceinline__ bool pdl_one_cluster() {
    uint32_t n;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return gridDim.x <= n;
}
__device__ __forceinline__ void pdl_release_early() {
    if (pdl_one_cluster()) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!pdl_one_cluster()) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------- fences ----
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// -------------------------------------------------------------- atomics ----
__device__ __forceinline__ void red_add_v4f32(void* p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};"
                 :
                 : "l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_f64(void* p, double a) {
    asm volatile("red.relaxed.gpu.global.add.f64 [%0], %1;" : : "l"(p), "d"(a) : "memory");
}

__device__ __forceinline__ void red_add_u32(void* p, uint32_t a) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" : : "l"(p), "r"(a) : "memory");
}

// ------------------------------------------------- L2 residency hints ----
// Cache policies for the bandwidth kernels: scratch that is written and read
// back within a step stays in L2 (evict_last) while the inputs and outputs
// that stream through once are the first to go (evict_first).
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_stream_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ld_input_v4_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint4 ld_relaxed_v4_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol)
                 : "memory");
    return v;
}

__device__ __forceinline__ void ld_relaxed_v2u64_hint(const void* p, uint64_t pol, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.L2::cache_hint.v2.u64 {%0,%1}, [%2], %3;"
                 : "=l"(a), "=l"(b)
                 : "l"(p), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_relaxed_v4_hint(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.relaxed.gpu.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_relaxed_v2u64_hint(void* p, uint64_t a, uint64_t b, uint64_t pol) {
    asm volatile("st.relaxed.gpu.global.L2::cache_hint.v2.u64 [%0], {%1,%2}, %3;"
                 :
                 : "l"(p), "l"(a), "l"(b), "l"(pol)
                 : "memory");
}

// Plain (weak) vector store with a policy: outputs, and sentinel resets whose
// next reader is ordered after them by the credit chain (a fence or the
// kernel boundary), never a concurrent poll.
__device__ __forceinline__ void st_weak_v4_hint(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// ---------------------------------------------------------------- timer ----
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// %globaltimer read that waits for `dep` (a value produced by an earlier load):
// a predicate is computed from `dep` inside the same asm block and guards the
// timer read, so the stamp cannot be taken before that load has returned
// (a C++ branch on `dep` may be turned into a select that reads the timer
// first).  Diagnostics only.
__device__ __forceinline__ uint64_t globaltimer_after(uint64_t dep) {
    uint64_t t;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.eq.u64 p, %1, 0x5A5A5A5A5A5A5A5A;\n\t"
        "@p mov.u64 %0, 0;\n\t"
        "@!p mov.u64 %0, %%globaltimer;\n\t}"
        : "=l"(t)
        : "l"(dep));
    return t;
}

// ---------------------------------------------------------- LL packing ----
// One 16-byte payload vector (four 32-bit words) travels as two 16-byte LL
// lines; every 64-bit element carries {payload word (low), epoch (high)}.
// "Every Microsecond Matters", Sec. IV "LL" and Fig. 8 (2 x sizeof(T) per
// element in LL mode).
__device__ __forceinline__ uint64_t ll_word(uint32_t payload, uint32_t epoch) {
    return (uint64_t)payload | ((uint64_t)epoch << 32);
}

__device__ __forceinline__ void ll_store(void* line_pair, uint4 v, uint32_t epoch) {
    char* q = (char*)line_pair;
    st_relaxed_v2u64(q, ll_word(v.x, epoch), ll_word(v.y, epoch));
    st_relaxed_v2u64(q + 16, ll_word(v.z, epoch), ll_word(v.w, epoch));
}

// Loads the two LL lines; returns true when all four flags equal `epoch`.
__device__ __forceinline__ bool ll_load(const void* line_pair, uint32_t epoch, uint4& out) {
    const char* q = (const char*)line_pair;
    uint64_t a, b, c, d;
    ld_relaxed_v2u64(q, a, b);
    ld_relaxed_v2u64(q + 16, c, d);
    out.x = (uint32_t)a;
    out.y = (uint32_t)b;
    out.z = (uint32_t)c;
    out.w = (uint32_t)d;
    return ((uint32_t)(a >> 32) == epoch) & ((uint32_t)(b >> 32) == epoch) &
           ((uint32_t)(c >> 32) == epoch) & ((uint32_t)(d >> 32) == epoch);
}

// ---------------------------------------------------------- sentinel ----
// The sentinel is the all-ones bit pattern (a negative quiet NaN in every
// type), "Every Microsecond Matters", Sec. IV "Sentinel".  A vector has
// arrived when none of its atomic units still holds the sentinel: 32-bit
// words for binary32/bfloat16 pairs (each word is stored atomically), 64-bit
// words for binary64 (a binary64 value is only all-ones if it IS the
// sentinel).
constexpr uint32_t kSentinel32 = 0xFFFFFFFFu;

template <int kUnitBytes>
__device__ __forceinline__ bool sentinel_arrived(uint4 v) {
    if (kUnitBytes == 8) {
        const bool lo = (v.x & v.y) != kSentinel32;
        const bool hi = (v.z & v.w) != kSentinel32;
        return lo & hi;
    } else {
        return (v.x != kSentinel32) & (v.y != kSentinel32) & (v.z != kSentinel32) &
               (v.w != kSentinel32);
    }
}

__device__ __forceinline__ uint4 sentinel_vec() {
    return make_uint4(kSentinel32, kSentinel32, kSentinel32, kSentinel32);
}

// Scratch transport of one 16-byte vector with the element width that is
// single-copy atomic for the type: 4 x 32-bit, or 2 x 64-bit for binary64 (so
// a binary64 value is never observed half-written).
template <int kUnitBytes>
__device__ __forceinline__ void st_scratch(void* p, uint4 v) {
    if (kUnitBytes == 8) {
        st_relaxed_v2u64(p, (uint64_t)v.x | ((uint64_t)v.y << 32), (uint64_t)v.z | ((uint64_t)v.w << 32));
    } else {
        st_relaxed_v4(p, v);
    }
}

template <int kUnitBytes>
__device__ __forceinline__ uint4 ld_scratch(const void* p) {
    if (kUnitBytes == 8) {
        uint64_t a, b;
        ld_relaxed_v2u64(p, a, b);
        return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
    } else {
        return ld_relaxed_v4(p);
    }
}

// The same with an L2 policy (the bandwidth kernels).
template <int kUnitBytes>
__device__ __forceinline__ void st_scratch_hint(void* p, uint4 v, uint64_t pol) {
    if (kUnitBytes == 8) {
        st_relaxed_v2u64_hint(p, (uint64_t)v.x | ((uint64_t)v.y << 32), (uint64_t)v.z | ((uint64_t)v.w << 32), pol);
    } else {
        st_relaxed_v4_hint(p, v, pol);
    }
}

template <int kUnitBytes>
__device__ __forceinline__ uint4 ld_scratch_hint(const void* p, uint64_t pol) {
    if (kUnitBytes == 8) {
        uint64_t a, b;
        ld_relaxed_v2u64_hint(p, pol, a, b);
        return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
    } else {
        return ld_relaxed_v4_hint(p, pol);
    }
}

// ------------------------------------------------------- bounded waits ----
// Every spin is bounded: each 64th iteration reads %globaltimer.  Past the
// deadline the waiter records RRA_ERR_TIMEOUT (first writer wins) and gives
// up.  Once a wait has lasted kStatusAfterNs it also reads the status word,
// so that when another CTA has already recorded an error all CTAs of a failed
// call leave promptly; normal (short) waits never touch that shared line.
constexpr uint64_t kStatusAfterNs = 20000;

struct Waiter {
    uint64_t deadline;      // give up after this %globaltimer value
    uint64_t status_after;  // read the status word only after this value
    Ctrl* ctrl;
    int rank;
    int step;
    uint32_t spins;
};

__device__ __forceinline__ Waiter make_waiter(uint64_t start_ns, uint64_t timeout_ns, Ctrl* ctrl, int rank,
                                              int step) {
    return Waiter{start_ns + timeout_ns, start_ns + kStatusAfterNs, ctrl, rank, step, 0u};
}

static __device__ __noinline__ void record_error(Ctrl* ctrl, uint32_t code, int rank, int step) {
    if (atomicCAS(&ctrl->status, 0u, code) == 0u) {
        ctrl->err_rank = rank;
        ctrl->err_step = step;
        uint32_t* const mirror = ctrl->host_status;
        if (mirror != nullptr) *(volatile uint32_t*)mirror = code;  // visible to the host once the stream completes
    }
}

// Returns true if the caller must give up.
__device__ __forceinline__ bool waiter_expired(Waiter& w) {
    if ((++w.spins & 63u) != 0u) return false;
    const uint64_t now = globaltimer_ns();
    if (now > w.deadline) {
        record_error(w.ctrl, RRA_ERR_TIMEOUT, w.rank, w.step);
        return true;
    }
    return now > w.status_after && ld_relaxed_u32(&w.ctrl->status) != 0u;
}

// ----------------------------------------------------- dtype handling ----
// Element-wise sum of two 16-byte vectors in the running type, and the
// conversions between the transported vector and the running values.
template <typename T>
struct VecMath;

// binary32: four elements, binary32 running value.
template <>
struct VecMath<float> {
    static constexpr int kElems = 4;
    static constexpr int kUnitBytes = 4;
    struct Acc { float v[4]; };
    __device__ __forceinline__ static Acc load(uint4 x) {
        Acc a;
        a.v[0] = __uint_as_float(x.x); a.v[1] = __uint_as_float(x.y);
        a.v[2] = __uint_as_float(x.z); a.v[3] = __uint_as_float(x.w);
        return a;
    }
    __device__ __forceinline__ static void add(Acc& a, uint4 x) {
        a.v[0] = __fadd_rn(a.v[0], __uint_as_float(x.x));
        a.v[1] = __fadd_rn(a.v[1], __uint_as_float(x.y));
        a.v[2] = __fadd_rn(a.v[2], __uint_as_float(x.z));
        a.v[3] = __fadd_rn(a.v[3], __uint_as_float(x.w));
    }
    __device__ __forceinline__ static uint4 store(const Acc& a) {
        return make_uint4(__float_as_uint(a.v[0]), __float_as_uint(a.v[1]),
                          __float_as_uint(a.v[2]), __float_as_uint(a.v[3]));
    }
};

// bfloat16: eight elements, binary32 running value, one rounding at the end.
template <>
struct VecMath<__nv_bfloat16> {
    static constexpr int kElems = 8;
    static constexpr int kUnitBytes = 4;
    struct Acc { float v[8]; };
    __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    __device__ __forceinline__ static Acc load(uint4 x) {
        Acc a;
        a.v[0] = lo(x.x); a.v[1] = hi(x.x); a.v[2] = lo(x.y); a.v[3] = hi(x.y);
        a.v[4] = lo(x.z); a.v[5] = hi(x.z); a.v[6] = lo(x.w); a.v[7] = hi(x.w);
        return a;
    }
    __device__ __forceinline__ static void add(Acc& a, uint4 x) {
        a.v[0] = __fadd_rn(a.v[0], lo(x.x)); a.v[1] = __fadd_rn(a.v[1], hi(x.x));
        a.v[2] = __fadd_rn(a.v[2], lo(x.y)); a.v[3] = __fadd_rn(a.v[3], hi(x.y));
        a.v[4] = __fadd_rn(a.v[4], lo(x.z)); a.v[5] = __fadd_rn(a.v[5], hi(x.z));
        a.v[6] = __fadd_rn(a.v[6], lo(x.w)); a.v[7] = __fadd_rn(a.v[7], hi(x.w));
    }
    __device__ __forceinline__ static uint32_t pack(float l, float h) {
        __nv_bfloat162 b = __floats2bfloat162_rn(l, h);  // .x = low half, .y = high half
        return *reinterpret_cast<uint32_t*>(&b);
    }
    __device__ __forceinline__ static uint4 store(const Acc& a) {
        return make_uint4(pack(a.v[0], a.v[1]), pack(a.v[2], a.v[3]), pack(a.v[4], a.v[5]),
                          pack(a.v[6], a.v[7]));
    }
};

// binary64: two elements, binary64 running value.
template <>
struct VecMath<double> {
    static constexpr int kElems = 2;
    static constexpr int kUnitBytes = 8;
    struct Acc { double v[2]; };
    __device__ __forceinline__ static double d(uint32_t lo, uint32_t hi) {
        return __hiloint2double((int)hi, (int)lo);
    }
    __device__ __forceinline__ static Acc load(uint4 x) {
        Acc a;
        a.v[0] = d(x.x, x.y);
        a.v[1] = d(x.z, x.w);
        return a;
    }
    __device__ __forceinline__ static void add(Acc& a, uint4 x) {
        a.v[0] = __dadd_rn(a.v[0], d(x.x, x.y));
        a.v[1] = __dadd_rn(a.v[1], d(x.z, x.w));
    }
    __device__ __forceinline__ static uint4 store(const Acc& a) {
        return make_uint4((uint32_t)__double2loint(a.v[0]), (uint32_t)__double2hiint(a.v[0]),
                          (uint32_t)__double2loint(a.v[1]), (uint32_t)__double2hiint(a.v[1]));
    }
};

// ------------------------------------------------- user input / output ----
// Input vector `vec` of a rank's buffer; elements at or beyond `count` read
// as zero (never the sentinel).
template <typename T>
__device__ __forceinline__ uint4 load_input(const void* base, uint32_t vec, uint64_t count) {
    constexpr int VE = VecMath<T>::kElems;
    const uint64_t e0 = (uint64_t)vec * VE;
    if (e0 + VE <= count) return ld_input_v4((const char*)base + (uint64_t)vec * kVecBytes);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    const int n = (int)(count - e0);
    if (sizeof(T) == 2) {
        const uint16_t* s = (const uint16_t*)base + e0;
        for (int i = 0; i < n; ++i) w[i >> 1] |= (uint32_t)s[i] << (16 * (i & 1));
    } else if (sizeof(T) == 4) {
        const uint32_t* s = (const uint32_t*)base + e0;
        for (int i = 0; i < n; ++i) w[i] = s[i];
    } else {
        const uint32_t* s = (const uint32_t*)base + 2 * e0;
        for (int i = 0; i < 2 * n; ++i) w[i] = s[i];
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// load_input with an L2 policy for the full vectors (the ragged tail is read
// as by load_input).
template <typename T>
__device__ __forceinline__ uint4 load_input_hint(const void* base, uint32_t vec, uint64_t count, uint64_t pol) {
    constexpr int VE = VecMath<T>::kElems;
    if ((uint64_t)vec * VE + VE <= count) return ld_input_v4_hint((const char*)base + (uint64_t)vec * kVecBytes, pol);
    return load_input<T>(base, vec, count);
}

// Output vector `vec`; only elements below `count` are written.
template <typename T>
__device__ __forceinline__ void store_output(void* base, uint32_t vec, uint64_t count, uint4 v) {
    constexpr int VE = VecMath<T>::kElems;
    const uint64_t e0 = (uint64_t)vec * VE;
    if (e0 + VE <= count) {
        st_output_v4((char*)base + (uint64_t)vec * kVecBytes, v);
        return;
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const int n = (int)(count - e0);
    if (sizeof(T) == 2) {
        uint16_t* d = (uint16_t*)base + e0;
        for (int i = 0; i < n; ++i) d[i] = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
    } else if (sizeof(T) == 4) {
        uint32_t* d = (uint32_t*)base + e0;
        for (int i = 0; i < n; ++i) d[i] = w[i];
    } else {
        uint32_t* d = (uint32_t*)base + 2 * e0;
        for (int i = 0; i < 2 * n; ++i) d[i] = w[i];
    }
}

// store_output with an L2 policy for full vectors.
template <typename T>
__device__ __forceinline__ void store_output_hint(void* base, uint32_t vec, uint64_t count, uint4 v, uint64_t pol) {
    constexpr int VE = VecMath<T>::kElems;
    if ((uint64_t)vec * VE + VE <= count) {
        st_weak_v4_hint((char*)base + (uint64_t)vec * kVecBytes, v, pol);
        return;
    }
    store_output<T>(base, vec, count, v);
}

}  // namespace rra

