// Kernel attributes of the cluster kernels, set once per process.
#ifndef RRA_KERNEL_ATTRS_H
#define RRA_KERNEL_ATTRS_H

#include <cuda_runtime.h>

#include <mutex>
#include <vector>

namespace rra {

// Opts kernel `k` in to `smem_bytes` of dynamic shared memory and to
// clusters of up to 16 CTAs.  The attributes are process-wide, so each
// kernel is configured once; the record of configured kernels is one for
// the whole library (an inline function's statics are shared by every
// translation unit) and guarded by a mutex, since calls on different
// communicators may launch from several host threads.
inline cudaError_t configure_cluster_kernel(const void* k, int smem_bytes) {
    static std::mutex mu;
    static std::vector<const void*> done;
    std::lock_guard<std::mutex> g(mu);
    for (const void* d : done)
        if (d == k) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done.push_back(k);
    return cudaSuccess;
}

}  // namespace rra

#endif  // RRA_KERNEL_ATTRS_H
