// host_cache.h -- per-device host-side caches of libsmoe.so (internal).
//
// The SM count and each kernel's raised dynamic shared-memory limit belong to
// a device, so a process that drives several GPUs keeps one entry per device.
// Entries are atomics (readers take no lock); raising a limit is serialised so
// the attribute a kernel ends up with is the largest one asked for.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace smoe {

constexpr int kMaxCachedDevices = 64;

// The current device as a cache index, or -1 when it cannot be read or lies
// past kMaxCachedDevices (callers then query without caching).
inline int cache_slot() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxCachedDevices) return -1;
    return d;
}

// The dynamic shared-memory limit a kernel has been raised to, per device
// (zero until the first raise; objects of static storage start zeroed).
using SmemLimits = std::atomic<int>[kMaxCachedDevices];

inline std::mutex &smem_limit_mutex() {
    static std::mutex m;
    return m;
}

// Make `kernel` launchable with `bytes` of dynamic shared memory on the
// current device: raises its limit once per device (the limit only grows).
template <typename Kernel>
cudaError_t allow_dynamic_smem(Kernel kernel, SmemLimits &limits, int bytes) {
    const int d = cache_slot();
    if (d >= 0 && limits[d].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    std::lock_guard<std::mutex> lock(smem_limit_mutex());
    const int have = d >= 0 ? limits[d].load(std::memory_order_relaxed) : 0;
    if (have >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && d >= 0) limits[d].store(bytes, std::memory_order_release);
    return e;
}

}  // namespace smoe
