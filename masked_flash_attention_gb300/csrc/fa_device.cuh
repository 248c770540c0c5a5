// fa_device.cuh -- device helpers shared by the scheduler and attention kernels:
// sequence geometry, the pair rules, the logit transform and the error word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace mfa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRowInf = 0x7fffffff;        // top-k: key never dropped
constexpr int kRowNever = (int)0x80000000; // top-k: key never kept

__device__ __forceinline__ int seq_qlen(const Params& p, int b) {
  return p.cu_q ? (p.cu_q[b + 1] - p.cu_q[b]) : p.Sq;
}
__device__ __forceinline__ int seq_klen(const Params& p, int b) {
  if (p.cache_len) return __ldg(p.cache_len + b) + seq_qlen(p, b);  // cached + active keys
  return p.cu_k ? (p.cu_k[b + 1] - p.cu_k[b]) : p.Sk;
}

// n / f.d for 0 <= n < 2^31 (see FastDiv).
__device__ __forceinline__ int fast_div(int n, const FastDiv& f) {
  return f.d == 1 ? n : (int)(__umulhi((uint32_t)n, f.mul) >> f.shr);
}

// Record the first device fault; later ones are dropped.
__device__ __forceinline__ void record_error(const Params& p, uint32_t code, uint32_t info) {
  if (atomicCAS(&p.ws->error, 0u, code) == 0u) atomicExch(&p.ws->error_info, info);
}

// True when sequence b's lengths, read from device memory, do not fit the
// sizes the host planned for (an item of such a sequence is skipped and the
// fault recorded, so nothing indexes with them).
__device__ __forceinline__ bool seq_lengths_bad(const Params& p, int b, int q_len, int kv_len) {
  bool bad = q_len < 0 || kv_len < 0 || q_len > p.Sq || kv_len > p.Sk;
  if (p.cu_q) bad |= p.cu_q[b] < 0 || (int64_t)p.cu_q[b + 1] > p.tot_q;
  if (p.cu_k && !p.block_table) bad |= p.cu_k[b] < 0 || (int64_t)p.cu_k[b + 1] > p.tot_k;
  if (p.cache_len) {  // two-source form: cached rows within the cache, appended rows too
    const int64_t lc = __ldg(p.cache_len + b);
    bad |= lc < 0 || lc > p.cache_cap || lc + q_len > p.Sk || (p.append && lc + q_len > p.cache_cap);
  }
  return bad;
}

// Query-row span [i0, i1] (inclusive, unclipped) of row tile `rt`.  For the
// decode path rows are packed (query, head-in-group) with `pack` = Hq/Hkv.
__device__ __forceinline__ void tile_rows(const Params& p, int rt, int& i0, int& i1) {
  if (p.path == FA_PATH_DECODE) {
    int P0 = rt * kDecodeRows;
    i0 = P0 / p.G;
    i1 = (P0 + kDecodeRows - 1) / p.G;
  } else {
    i0 = rt * p.rows_per_tile;
    i1 = i0 + p.rows_per_tile - 1;
  }
}

// The pair rules (bottom-right causal, sliding window, key bound) for one pair.
__device__ __forceinline__ bool pair_allowed(const Params& p, int i, int j, int off, int kv_len) {
  bool ok = (j >= 0) & (j < kv_len);
  if (p.causal) ok &= (j <= i + off);
  if (p.wl >= 0) ok &= (j >= i + off - p.wl);
  if (p.wr >= 0) ok &= (j <= i + off + p.wr);
  return ok;
}

// Inclusive key range any row of [i0, i1] may see under the pair rules.
__device__ __forceinline__ void key_range(const Params& p, int i0, int i1, int off, int kv_len,
                                          int& jlo, int& jhi) {
  jlo = 0;
  jhi = kv_len - 1;
  if (p.causal) jhi = min(jhi, i1 + off);
  if (p.wl >= 0) jlo = max(jlo, i0 + off - p.wl);
  if (p.wr >= 0) jhi = min(jhi, i1 + off + p.wr);
}

// True when every pair of rows [i0, i1] x keys [kj0, kj1] passes the pair rules.
__device__ __forceinline__ bool tile_all_allowed(const Params& p, int i0, int i1, int kj0, int kj1,
                                                 int off, int kv_len) {
  bool ok = (kj1 < kv_len);
  if (p.causal) ok &= (kj1 <= i0 + off);
  if (p.wl >= 0) ok &= (kj0 >= i1 + off - p.wl);
  if (p.wr >= 0) ok &= (kj1 <= i0 + off + p.wr);
  return ok;
}

__device__ __forceinline__ float fast_exp2(float x);

// Soft-capped logit in log2 units: cap * tanh(x / cap) * log2(e), with
// tanh(y) = sign(y) (1 - t) / (1 + t), t = 2^(-2 log2(e) |y|) -- one hardware
// exp2 and one fast division instead of a full-precision tanh and divide.
// For small |y| the rounding of 1 - t costs about 1e-7 relative to 1, i.e.
// ~1e-6 in the logit at cap 30: far below the bf16 rounding of P.
__device__ __forceinline__ float softcap_log2(float x, float cap, float inv_cap) {
  const float y = x * inv_cap;
  const float t = fast_exp2(-2.f * kLog2e * fabsf(y));
  const float th = __fdividef(1.f - t, 1.f + t);
  return copysignf(th, y) * (cap * kLog2e);
}

// Full logit transform of one raw dot product `s` for (sequence b, q-head h,
// query row i, key j), returned in log2 units (x * log2 e), -inf if dropped:
// scale, soft-cap, ALiBi, pair rules, dense mask or top-k (keep test + bias).
__device__ __forceinline__ float logit_log2(const Params& p, float s, int b, int h, int i, int j,
                                            int off, int kv_len) {
  if (!pair_allowed(p, i, j, off, kv_len)) return -INFINITY;
  float x = (p.softcap > 0.f) ? softcap_log2(s * p.scale, p.softcap, p.inv_softcap) : s * p.scale_log2;
  if (p.alibi) x -= __ldg(p.alibi + h) * kLog2e * (float)abs(i + off - j);
  if (p.mask_kind == FA_MASK_DENSE) {
    const float* m = p.mask + (int64_t)(p.m_nb > 1 ? b : 0) * p.m_sb +
                     (int64_t)(p.m_nh > 1 ? h : 0) * p.m_sh + (int64_t)i * p.m_sq +
                     (int64_t)j * p.m_sk;
    x += __ldg(m) * kLog2e;
  } else if (p.mask_kind == FA_MASK_TOPK) {
    int64_t bh = (int64_t)b * p.Hq + h;
    int e = __ldg(p.topk_e + bh * p.Sk + j);
    if (!(i < e)) return -INFINITY;
    x += __ldg(p.z + (int64_t)b * p.z_sb + (int64_t)h * p.z_sh + (int64_t)j * p.z_sk) * kLog2e;
  }
  return x;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mfa
