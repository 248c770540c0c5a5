// host_util.h -- host-side helpers shared by the launchers.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

namespace mfa {

// Set a kernel's dynamic shared-memory limit once per device (the attribute
// persists for the process), so that repeated launches pay no host call.  The
// kernel is a template argument, so each kernel has its own flag (kernels of
// one signature share a function-pointer type).
template <auto kern>
inline cudaError_t ensure_smem_attr(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

}  // namespace mfa
