// noalloc.cu -- fa_fwd_noalloc: the same forward as fa_fwd, for callers that
// cannot allocate device memory, with its scratch (tile work list, scheduler
// counters, split-KV partial results, error word) in one static device array
// that the library owns.
//
// Who needs this: code that runs where cudaMalloc is off limits, e.g. inside
// an allocator-free inference runtime that hands out only pre-sized I/O
// buffers, a plugin whose host forbids device allocations after start-up, or a
// caller that must not touch the allocator at all on its latency path.  They
// pass inputs and outputs as usual; the library supplies the scratch.
//
// Costs and limits: every GPU that loads the library holds the array
// (kNoAllocScratchBytes) until the process exits; problems whose scratch need
// is larger are rejected with FA_ERR_WORKSPACE; all calls share the array, so
// calls that overlap on the GPU (different streams, different threads) race
// on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code `g_scratch` is only a host-side stand-in
// for the symbol, never a device address: the device address is obtained with
// cudaGetSymbolAddress, per device, below.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_dev[kMaxDevices];  // device address of g_scratch, per device
std::mutex g_setup_mutex;

// One-time set-up per device (with that device current): look up the device
// address of the static scratch.  Returns nullptr on failure.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_dev[dev] = p;
  }
  return g_scratch_dev[dev];
}

}  // namespace

extern "C" int fa_fwd_noalloc(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                              const fa_tensor* out, const fa_tensor* lse,
                              const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                              const fa_tensor* block_table, const fa_mask* mask,
                              int32_t window_left, int32_t window_right, float softcap,
                              float scale, int32_t causal, const fa_opts* opts) {
  if (!opts) return FA_ERR_INVALID_ARG;
  fa_opts o = *opts;
  o.workspace = nullptr;
  o.workspace_bytes = 0;
  size_t need = 0;
  int rc = fa_fwd_workspace_size(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask,
                                 window_left, window_right, softcap, scale, causal, &o, &need);
  if (rc != FA_OK) return rc;
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;  // beyond the static scratch
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  void* scratch = scratch_address(dev);
  if (!scratch) return FA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(o.stream);
  // the array keeps the previous call's contents: the error word must start
  // at zero (the scheduler counters are cleared by every forward call)
  if (cudaMemsetAsync(scratch, 0, sizeof(mfa::WsHeader), st) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  o.workspace = scratch;
  o.workspace_bytes = kNoAllocScratchBytes;
  return fa_fwd(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, window_left,
                window_right, softcap, scale, causal, &o);
}
