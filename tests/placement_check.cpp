// Host-only checks of the bulk-copy placement rule (placement.h) against a
// fake memory map: which source sets may be read by bulk copies with cluster
// multicast, where the checked range ends, and what the cache of passing sets
// remembers.  Built with g++ by tests/test_placement_cpu.py; no CUDA.
#include <cstdint>
#include <cstdio>
#include <utility>
#include <vector>

#include "placement.h"

namespace {

// Device memory of the current GPU: a list of [lo, hi) ranges; every other
// address is something else (host, another GPU, managed).
struct FakeMap {
    std::vector<std::pair<uintptr_t, uintptr_t>> device;
    int queries = 0;
    bool operator()(const void* p) {
        ++queries;
        const uintptr_t a = (uintptr_t)p;
        for (const auto& r : device)
            if (a >= r.first && a < r.second) return true;
        return false;
    }
};

int failures = 0, checks = 0;

void check(bool ok, const char* what) {
    ++checks;
    if (!ok) {
        ++failures;
        std::printf("FAIL %s\n", what);
    }
}

const void* at(uintptr_t a) { return (const void*)a; }

}  // namespace

int main() {
    using rra::placement::SourceCache;
    FakeMap map;
    // four device buffers of 4096 bytes, 1 MiB apart; one of 100 and one of 112 bytes
    for (int r = 0; r < 4; ++r) map.device.push_back({0x100000u + 0x100000u * r, 0x100000u + 0x100000u * r + 4096});
    map.device.push_back({0x900000u, 0x900000u + 100});
    map.device.push_back({0xA00000u, 0xA00000u + 112});
    const void* dev4[4] = {at(0x100000), at(0x200000), at(0x300000), at(0x400000)};
    auto q = [&](SourceCache& c, bool other, const void* const* src, int n, size_t bytes) {
        return rra::placement::bulk_sources_local(c, other, src, n, bytes, map);
    };

    {   // every source in device memory: passes after two queries per source
        SourceCache c;
        map.queries = 0;
        check(q(c, false, dev4, 4, 4096), "four device buffers, full length");
        check(map.queries == 8, "first and last byte of each source queried");
        check(q(c, false, dev4, 4, 4096), "the same set again");
        check(map.queries == 8, "a remembered set is not queried again");
        check(q(c, false, dev4, 4, 2048), "the same set, fewer bytes");
        check(map.queries == 8, "fewer bytes: still no query");
        check(!q(c, false, dev4, 4, 4097), "one byte past the buffers: the last vector leaves device memory");
        check(map.queries > 8, "more bytes than remembered: queried again");
        check(q(c, false, dev4, 3, 4096), "a three-rank prefix passes on its own queries");
    }
    {   // the range read is rounded up to a whole 16-byte vector
        SourceCache c;
        const void* b100[1] = {at(0x900000)};
        const void* b112[1] = {at(0xA00000)};
        check(!q(c, false, b100, 1, 100), "100 bytes in a 100-byte buffer: the copy reads 112");
        check(q(c, false, b112, 1, 100), "100 bytes in a 112-byte buffer");
        check(q(c, false, b112, 1, 112), "112 bytes in a 112-byte buffer");
        check(!q(c, false, b112, 1, 113), "113 bytes read 128");
    }
    {   // one source elsewhere, or missing: no bulk copies
        SourceCache c;
        const void* mixed[4] = {dev4[0], dev4[1], at(0x7f0000000000ull), dev4[3]};
        check(!q(c, false, mixed, 4, 64), "one source in host memory");
        const void* hole[4] = {dev4[0], nullptr, dev4[2], dev4[3]};
        check(!q(c, false, hole, 4, 64), "a null source");
        const void* inside[2] = {at(0x100000 + 4000), dev4[1]};
        check(!q(c, false, inside, 2, 200), "a source that starts in device memory and runs past it");
    }
    {   // another GPU in use, or arguments out of range: no queries at all
        SourceCache c;
        map.queries = 0;
        check(!q(c, true, dev4, 4, 64), "another GPU in use");
        check(!q(c, false, dev4, 0, 64), "no ranks");
        check(!q(c, false, dev4, 4, 0), "no bytes");
        check(!q(c, false, nullptr, 4, 64), "no source array");
        const void* many[65];
        for (int r = 0; r < 65; ++r) many[r] = dev4[r % 4];
        check(!q(c, false, many, 65, 64), "more ranks than a bulk-copy kernel serves");
        check(map.queries == 0, "none of these queried the map");
        check(q(c, false, many, 64, 64), "sixty-four ranks");
        check(!q(c, true, many, 64, 64), "another GPU in use outranks a remembered set");
    }
    {   // the cache holds the last 8 sets
        SourceCache c;
        const void* sets[9][1];
        for (int k = 0; k < 9; ++k) sets[k][0] = at(0x100000 + 16 * k);
        for (int k = 0; k < 9; ++k) check(q(c, false, sets[k], 1, 16), "nine single-source sets");
        map.queries = 0;
        check(q(c, false, sets[8], 1, 16), "the newest set");
        check(map.queries == 0, "the newest set is remembered");
        check(q(c, false, sets[1], 1, 16), "the second set");
        check(map.queries == 0, "the second set is remembered");
        check(q(c, false, sets[0], 1, 16), "the first set");
        check(map.queries == 2, "the first set was overwritten by the ninth");
    }
    {   // sets are matched by address: clear() forgets them
        SourceCache c;
        check(q(c, false, dev4, 4, 4096), "the set passes");
        FakeMap saved = map;
        map.device.clear();  // the buffers freed, their addresses now something else
        check(q(c, false, dev4, 4, 4096), "remembered by address alone");
        c.clear();
        check(!q(c, false, dev4, 4, 4096), "after clear() the set is queried and fails");
        map = saved;
    }
    std::printf("%d checks, %d failed\n", checks, failures);
    return failures == 0 ? 0 : 1;
}
