// Where the bulk-copy push may read its sources, as plain host C++.
//
// The bulk-copy push (cp.async.bulk with .multicast::cluster) reads each
// rank's input straight from the caller's buffer.  Loads with cluster
// multicast are kept to single-GPU processes reading this GPU's own device
// memory, so a call may use the push only when
//   (a) the process holds no active context on another GPU, and
//   (b) every byte the copies read lies in device memory of the current GPU.
// Copies move whole 16-byte vectors, so the range checked for a source is
// `bytes` rounded up to a whole vector; its first and its last byte are
// queried.
//
// The device query is a parameter (the library passes one built on
// cudaPointerGetAttributes), so the rule compiles and is tested without CUDA.
#ifndef RRA_PLACEMENT_H
#define RRA_PLACEMENT_H

#include <array>
#include <cstddef>

namespace rra {
namespace placement {

constexpr int kMaxRanks = 64;      // ranks a bulk-copy kernel serves
constexpr size_t kVecBytes = 16;   // bulk copies move whole 16-byte vectors

// Source sets that passed the check, matched afterwards by address alone;
// the newest overwrites the oldest.
struct SourceCache {
    struct Entry {
        int n = 0;
        size_t bytes = 0;
        const void* ptr[kMaxRanks] = {};
    };
    std::array<Entry, 8> entry{};
    int next = 0;
    void clear() { *this = SourceCache{}; }
};

// True when bulk copies may read `bytes` from each of src[0..n-1].
// `other_gpu_in_use`: the process drives another GPU (or that is unknown).
// `on_device(p)`: address p lies in device memory of the current GPU.
// A set already in `cache` with the same n and pointers and at least as many
// bytes passes without a query; a set that passes the queries is added.
template <class OnDevice>
bool bulk_sources_local(SourceCache& cache, bool other_gpu_in_use, const void* const src[], int n, size_t bytes,
                        OnDevice&& on_device) {
    if (src == nullptr || n < 1 || n > kMaxRanks || bytes == 0) return false;
    if (other_gpu_in_use) return false;
    for (const auto& e : cache.entry) {
        if (e.n != n || bytes > e.bytes) continue;
        bool same = true;
        for (int r = 0; r < n && same; ++r) same = e.ptr[r] == src[r];
        if (same) return true;
    }
    const size_t span = (bytes + kVecBytes - 1) / kVecBytes * kVecBytes;
    for (int r = 0; r < n; ++r) {
        if (src[r] == nullptr) return false;
        if (!on_device(src[r]) || !on_device((const char*)src[r] + (span - 1))) return false;
    }
    auto& e = cache.entry[(size_t)cache.next];
    cache.next = (cache.next + 1) % (int)cache.entry.size();
    e.n = n;
    e.bytes = bytes;
    for (int r = 0; r < n; ++r) e.ptr[r] = src[r];
    return true;
}

}  // namespace placement
}  // namespace rra

#endif  // RRA_PLACEMENT_H
