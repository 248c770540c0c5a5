// host_util.h -- host-side helpers shared by the launchers.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda.h>
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

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); null when the driver does not provide it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    cudaGetLastError();
  });
  return fn;
}

// 4-D map of 2-byte elements (bf16, or fp16 when f16) {d, heads, rows, outer}
// with box {box_d, 1, box_rows, 1}.  Strides are in elements (head, row,
// outer).  False when the driver rejects the layout (alignment, strides) or
// has no encoder.
inline bool encode_4d_bf16(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int64_t outer,
                           int64_t s_h, int64_t s_row, int64_t s_outer, int box_d, int box_rows,
                           CUtensorMapSwizzle swz, CUtensorMapL2promotion l2, bool f16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[3] = {(cuuint64_t)s_h * 2, (cuuint64_t)s_row * 2, (cuuint64_t)s_outer * 2};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map of 2-byte elements {cols, rows} (row stride s_row elements) with
// box {box_cols, 1} and 128-byte swizzle, for tile::gather4 loads of single
// rows.  False when the driver rejects the layout or has no encoder.
inline bool encode_rows_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t s_row,
                             int box_cols, bool f16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)s_row * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mfa
