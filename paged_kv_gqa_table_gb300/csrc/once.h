// once.h -- per-device set-up on the host that stays correct when several host
// threads make their first call on a device at the same time.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace pkv {

constexpr int kMaxDevices = 64;

// Runs fn() (returning cudaError_t) for device `dev` until it first succeeds;
// later calls return cudaSuccess at the cost of one acquire load.  Concurrent
// first calls are serialised by `mu`, so fn() never runs twice at once.
template <typename Fn>
cudaError_t once_per_device(std::atomic<bool> (&done)[kMaxDevices], std::mutex& mu, int dev, Fn&& fn) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = fn();
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
}

// SM count of device `dev`, queried once and cached (an idempotent value, so
// concurrent first queries may both store it).
inline cudaError_t device_sm_count(int dev, int* out) {
    static std::atomic<int> cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidValue;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return cudaSuccess;
}

// The current device's SM count.
inline cudaError_t current_device_sm_count(int* out) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return device_sm_count(dev, out);
}

}  // namespace pkv
