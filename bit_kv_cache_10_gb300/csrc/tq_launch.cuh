// Per-kernel setup calls done once per device instead of before every launch.
//
// Raising a kernel's dynamic shared-memory limit and asking for its cluster
// occupancy are host calls into the runtime that cost a microsecond or more
// each; a decode call's whole host side is a few microseconds.  Each launch
// function keeps one KernelMemo (a function-local static, so one per kernel
// instantiation) whose bit d records that device d has the limit set, and the
// device's occupancy.  The limit belongs to the device's context: if the
// context was reset since it was set, or a launch needs more shared memory
// than the limit set first (the quantize kernels' size depends on the code
// widths), the launch is refused, and launch_with_limit sets the limit to this
// launch's size and launches once more.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

namespace tq {

struct KernelMemo {
  static constexpr int kDevices = 64;
  std::atomic<unsigned long long> limit_set{0};  // bit d: the limit is set on device d
  std::atomic<int> fit[kDevices] = {};           // occupancy + 1 on device d, 0 = not asked yet
};

// Device ordinal of the calling thread, -1 on error.
inline int current_device() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

// Sets the kernel's dynamic shared-memory limit on device `dev` unless the memo
// has it (always when `force`).  False on a CUDA error.
template <typename Kern>
bool ensure_smem_limit(Kern kern, int bytes, KernelMemo& memo, int dev, bool force = false) {
  const unsigned long long bit = dev >= 0 && dev < KernelMemo::kDevices ? 1ull << dev : 0ull;
  if (!force && bit != 0 && (memo.limit_set.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  memo.limit_set.fetch_or(bit, std::memory_order_release);
  return true;
}

// Clusters of `cfg` resident at once on device `dev` (asked once per device), or
// -1 on a CUDA error.  The limit must be set.
template <typename Kern>
int cluster_fit(Kern kern, const cudaLaunchConfig_t& cfg, KernelMemo& memo, int dev) {
  const bool cached = dev >= 0 && dev < KernelMemo::kDevices;
  if (cached) {
    const int f = memo.fit[dev].load(std::memory_order_acquire);
    if (f > 0) return f - 1;
  }
  int fit = 0;
  if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess) return -1;
  if (cached) memo.fit[dev].store(fit + 1, std::memory_order_release);
  return fit;
}

// cudaLaunchKernelEx after the limit is ensured; a launch refused while the memo
// claimed the limit (a reset context) sets it again and is retried once.
template <typename Kern, typename... Args>
cudaError_t launch_with_limit(Kern kern, int bytes, KernelMemo& memo, int dev, const cudaLaunchConfig_t& cfg,
                              Args... args) {
  if (!ensure_smem_limit(kern, bytes, memo, dev)) return cudaErrorInvalidValue;
  if (cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess) return cudaSuccess;
  (void)cudaGetLastError();  // the refused launch's error (not sticky)
  if (!ensure_smem_limit(kern, bytes, memo, dev, true)) return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace tq
