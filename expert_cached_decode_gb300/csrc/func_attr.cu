// Per-device kernel attributes.  A kernel's dynamic shared-memory limit is a
// property of the kernel on one device: a process that launches on several
// GPUs must raise it on each.  The raised value is remembered per (device,
// kernel) under a lock, so the attribute call happens once per device and
// never while a launch on another thread is being prepared with a stale view.
#include <map>
#include <mutex>
#include <utility>

#include "internal.h"

namespace moe {

cudaError_t ensure_dyn_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = raised[std::make_pair(dev, func)];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  have = bytes;
  return cudaSuccess;
}

}  // namespace moe
