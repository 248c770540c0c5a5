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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code `g_scratch` is only a host-side stand-in
// for the symbol, never a device address: the device address is obtained with
// cudaGetSymbolAddress, per device, below.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

// Driver calls reached through the runtime's entry-point query (no link
// against libcuda): the current context and its process-unique ID.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(a);
      f.get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    cudaGetLastError();
  });
  return f;
}

constexpr int kMaxDevices = 64;
// Device address of g_scratch per device, with the ID of the context it was
// looked up in.  The module (and so the array) is loaded again, possibly at
// another address, when a device's primary context is destroyed and created
// anew (cudaDeviceReset, or releasing the primary context), so the address is
// only reused while the current context is the same one.
struct ScratchSlot {
  unsigned long long ctx_id = 0;  // 0: not looked up yet
  void* addr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the static scratch for the current context of device
// `dev` (set-up once per device and context, with that device current).
// Returns nullptr on failure.
void* scratch_address(int dev) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& s = g_slots[dev];
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  const bool have_ctx = f.get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr;
  if (have_ctx && f.get_id(ctx, &id) == CUDA_SUCCESS && id != 0 && id == s.ctx_id && s.addr) return s.addr;
  // look the address up (this also makes the runtime bind the device's
  // primary context when the thread has none yet), then record the context
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    s = ScratchSlot{};
    return nullptr;
  }
  ctx = nullptr;
  id = 0;
  if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx || f.get_id(ctx, &id) != CUDA_SUCCESS || id == 0) {
    s = ScratchSlot{};
    return nullptr;
  }
  s.ctx_id = id;
  s.addr = p;
  return p;
}

}  // namespace

extern "C" int fa_fwd_noalloc(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                              const fa_tensor* out, const fa_tensor* lse,
                              const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                              const fa_tensor* block_table, const fa_mask* mask,
                              int32_t window_left, int32_t window_right, float softcap,
                              float scale, int32_t causal, const fa_opts* opts) {
  if (!opts) return FA_ERR_INVALID_ARG;
  // the device error word is cleared by every call and cannot be read back,
  // so a device-side value check could never be reported: refuse it
  if (opts->debug_flags & FA_DEBUG_VALIDATE) return FA_ERR_UNSUPPORTED;
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
  // the array keeps the previous call's contents: the error word and the
  // tail-split counts must start at zero (the scheduler counters are cleared
  // by every forward call)
  if (cudaMemsetAsync(scratch, 0, mfa::kWsHeadBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  o.workspace = scratch;
  o.workspace_bytes = kNoAllocScratchBytes;
  // no profiler ranges on this path: it calls nothing beyond the CUDA runtime
  const bool trace = mfa::g_trace_ranges;
  mfa::g_trace_ranges = false;
  const int r = fa_fwd(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, window_left,
                       window_right, softcap, scale, causal, &o);
  mfa::g_trace_ranges = trace;
  return r;
}
