// backward_sm103.cu -- the backward pass on the 5th-generation tensor cores
// (dK/dV kernel further down).  dQ: one CTA per (sequence, q-head, 128-row
// query tile), for every key tile its rows can see
//   S  = Q K^T,   dP = dO V^T                 (tcgen05, TMEM accumulators)
//   dS = P * (dP - Delta) * dx/ds,  P = exp(x - LSE)   (one thread per row)
//   dQ += dS K                                (tcgen05, dS read from TMEM)
// the same products as the warp-level dq kernel (backward.cu), with the
// operand layouts of the forward kernel: Q, dO, K and V tiles arrive by TMA
// (128-byte swizzle, K-major for S and dP); K is also the MN-major B operand
// of dQ += dS K, as V is for the forward's PV; dS is packed in place of the S
// it came from, as the forward packs P.
//
// Thread 0 issues the TMA copies and the MMAs; all 512 threads turn S and dP
// into dS: warpgroup k takes key columns [32 k, 32 k + 32) of every row (a
// warp reaches TMEM lanes 32 (warp % 4) ...), so thread (k, r) owns row r,
// 32 keys.  TMEM: S [0, 128), dS [128, 192), dP [256, 384), dQ [384, 384 + D).
// K/V tiles in two buffers.  Order per key tile t: S(t), dP(t) -> rows ->
// dQ(t) += dS(t) K(t); the next tile's S and dP are issued once every row has
// read S(t) and dP(t) (right after dQ(t)), and the copy of tile t + 2 into
// tile t's buffer waits for the commit that follows dQ(t).  Every wait is
// bounded (FA_ERR_DEVICE_TIMEOUT on expiry).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fa_device.cuh"
#include "host_util.h"
#include "tc_sm103.cuh"

namespace mfa {

namespace {

constexpr int kTcRows = 128;   // query rows per CTA (TMEM lanes)
constexpr int kTcKeys = 128;   // keys per tile
constexpr uint32_t kTcCols = 512;

template <int D>
struct DqTcCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128-row tile
  static constexpr int kQ = 0, kDO = kTile;
  static constexpr int kKV = 2 * kTile;      // [2 buffers][K, V]
  static constexpr int kBar = kKV + 4 * kTile;
  static constexpr int kUsed = kBar + 256;
  // at least 116 KB, so that one CTA (and its 512 TMEM columns) sits on an SM
  static constexpr int kSmem = (kUsed > 116 * 1024 ? kUsed : 116 * 1024) + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ float tc_softcap_tanh(float x, float inv_cap) {
  const float y = x * inv_cap;
  const float t = fast_exp2(-2.f * kLog2e * fabsf(y));
  return copysignf(__fdividef(1.f - t, 1.f + t), y);
}

template <bool F16>
__device__ __forceinline__ uint32_t tc_pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(512, 1)
    dq_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using C = DqTcCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n_qt = (p.Sq + kTcRows - 1) / kTcRows;
  const int qt = (int)(blockIdx.x % n_qt);
  const int64_t r0 = blockIdx.x / n_qt;
  const int h = (int)(r0 % p.Hq), b = (int)(r0 / p.Hq);
  const int g = h / p.G;
  // lengths from device memory, checked against the planned sizes
  const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
  {
    bool bad = q_len < 0 || kv_len < 0 || q_len > p.Sq || kv_len > p.Sk;
    if (p.cu_q) bad |= p.cu_q[b] < 0 || (int64_t)p.cu_q[b + 1] > p.tot_q;
    if (p.cu_k) bad |= p.cu_k[b] < 0 || (int64_t)p.cu_k[b + 1] > p.tot_k;
    if (bad) return;  // the dK/dV kernel reports it
  }
  const int i0 = qt * kTcRows;
  if (i0 >= q_len) return;
  const int off = kv_len - q_len;
  int jlo, jhi;
  key_range(p, i0, min(i0 + kTcRows, q_len) - 1, off, kv_len, jlo, jhi);
  const int kb0 = jlo > 0 ? jlo / kTcKeys : 0;
  const int nkb = jhi >= jlo ? jhi / kTcKeys - kb0 + 1 : 0;
  const int wg = warp >> 2;                      // key columns [32 wg, 32 wg + 32)
  const int row = 32 * (warp & 3) + (tid & 31), i = i0 + row;  // this thread's query row

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* q_full = bars;         // Q and dO landed
  uint64_t* kv_full = bars + 1;    // [2] K/V buffer landed
  uint64_t* s_done = bars + 3;     // S and dP of a tile written
  uint64_t* ds_ready = bars + 4;   // dS of a tile written (512 threads)
  uint64_t* q_done = bars + 5;     // dQ MMA of a tile (and all before it) done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  if (tid == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(kv_full + 1, 1);
    tc::mbar_init(s_done, 1);
    tc::mbar_init(ds_ready, 512);
    tc::mbar_init(q_done, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTcCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t lane_base = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
  constexpr uint32_t kDSCol = 128, kDPCol = 256, kDQCol = 384;

  const int q_row0 = p.cu_q ? p.cu_q[b] : 0, q_b = p.cu_q ? 0 : b;
  const int k_row0 = p.cu_k ? p.cu_k[b] : 0, k_b = p.cu_k ? 0 : b;
  constexpr uint32_t idS = tc::idesc_bf16_f32(128, 128, false, false, F16);
  constexpr uint32_t idQ = tc::idesc_bf16_f32(128, D, false, true, F16);
  const uint32_t sQ = tc::smem_u32(smem + C::kQ), sDO = tc::smem_u32(smem + C::kDO);
  auto kv_base = [&](int buf) { return smem + C::kKV + buf * 2 * C::kTile; };
  auto load_kv = [&](int t) {
    unsigned char* dst = kv_base(t & 1);
    tc::mbar_arrive_expect_tx(kv_full + (t & 1), 2 * C::kTile);
    const int row_k = k_row0 + (kb0 + t) * kTcKeys;
    for (int c = 0; c < D / 64; ++c) {
      tc::tma_load_4d(dst + c * 16384, &tk, kv_full + (t & 1), c * 64, g, row_k, k_b);
      tc::tma_load_4d(dst + C::kTile + c * 16384, &tv, kv_full + (t & 1), c * 64, g, row_k, k_b);
    }
  };
  auto issue_s = [&](int t) {  // S(t) -> S, dP(t) -> dP
    const uint32_t ka = tc::smem_u32(kv_base(t & 1)), va = ka + C::kTile;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
      tc::mma_ss(tbase, tc::sdesc_sw128(sQ + o, 16, 1024), tc::sdesc_sw128(ka + o, 16, 1024), idS,
                 ks > 0 ? 1u : 0u);
      tc::mma_ss(tbase + kDPCol, tc::sdesc_sw128(sDO + o, 16, 1024), tc::sdesc_sw128(va + o, 16, 1024), idS,
                 ks > 0 ? 1u : 0u);
    }
    tc::mma_commit(s_done);
  };

  bool ok = true;
  if (tid == 0 && nkb > 0) {
    tc::tma_prefetch_desc(&tq);
    tc::tma_prefetch_desc(&tdo);
    tc::tma_prefetch_desc(&tk);
    tc::tma_prefetch_desc(&tv);
    tc::mbar_arrive_expect_tx(q_full, 2 * C::kTile);
    for (int c = 0; c < D / 64; ++c) {
      tc::tma_load_4d(smem + C::kQ + c * 16384, &tq, q_full, c * 64, h, q_row0 + i0, q_b);
      tc::tma_load_4d(smem + C::kDO + c * 16384, &tdo, q_full, c * 64, h, q_row0 + i0, q_b);
    }
    load_kv(0);
    if (nkb > 1) load_kv(1);
    ok = tc::mbar_wait(q_full, 0, abort_flag) && tc::mbar_wait(kv_full, 0, abort_flag);
    if (ok) {
      tc::fence_after_sync();
      issue_s(0);
    } else {
      *abort_flag = 1;
    }
  }
  // this row's LSE (log2 units) and Delta
  float lse2 = 0.f, dlt = 0.f;
  if (i < q_len) {
    const int64_t qrow = (int64_t)q_row0 + i;
    lse2 = __ldg(p.lse + (p.cu_q ? 0 : (int64_t)b * p.lse_sb) + (int64_t)h * p.lse_sh + qrow * p.lse_ss) * kLog2e;
    dlt = p.delta[p.cu_q ? (int64_t)h * p.tot_q + qrow : ((int64_t)b * p.Hq + h) * p.Sq + i];
  }
  const float slope2 = p.alibi ? __ldg(p.alibi + h) * kLog2e : 0.f;
  // the pair rules for this row as one interval of keys [jlo_i, jhi_i]
  int jlo_i = 0, jhi_i = kv_len - 1;
  if (i >= q_len) jhi_i = -1;
  if (p.causal) jhi_i = min(jhi_i, i + off);
  if (p.wl >= 0) jlo_i = max(jlo_i, i + off - p.wl);
  if (p.wr >= 0) jhi_i = min(jhi_i, i + off + p.wr);
  const bool plain = !(p.softcap > 0.f) && !p.alibi;  // logit = scale * s

  for (int t = 0; t < nkb; ++t) {
    // ---- the rows: S(t), dP(t) -> dS(t), this thread's 32 keys
    if (!ok || !tc::mbar_wait_spin(s_done, t & 1, abort_flag)) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    const int j0 = (kb0 + t) * kTcKeys;
    {
      const int c = wg;
      uint32_t sv[32], dv[32];
      tc::tmem_ld32(lane_base + 32 * c, sv);
      tc::tmem_ld32(lane_base + kDPCol + 32 * c, dv);
      tc::tmem_wait_ld();
      uint32_t pk[16];
      const int jb = j0 + 32 * c;  // key of column 0 of this thread's chunk
      if (plain) {
        const float nl = -lse2, ds_scale = p.scale;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float ds[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = jb + e + u;
            const bool in = (j >= jlo_i) & (j <= jhi_i);
            const float pe = in ? fast_exp2(fmaf(__uint_as_float(sv[e + u]), p.scale_log2, nl)) : 0.f;
            ds[u] = pe * (__uint_as_float(dv[e + u]) - dlt) * ds_scale;
          }
          pk[e >> 1] = tc_pack2<F16>(ds[0], ds[1]);
        }
      } else
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float ds[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = jb + e + u;
          const float s = __uint_as_float(sv[e + u]);
          float x = -INFINITY, dxds = 0.f;
          if ((j >= jlo_i) & (j <= jhi_i)) {
            if (p.softcap > 0.f) {
              const float th = tc_softcap_tanh(s * p.scale, p.inv_softcap);
              x = th * (p.softcap * kLog2e);
              dxds = p.scale * (1.f - th * th);
            } else {
              x = s * p.scale_log2;
              dxds = p.scale;
            }
            x -= slope2 * (float)abs(i + off - j);
          }
          const float pe = (x == -INFINITY) ? 0.f : fast_exp2(x - lse2);
          ds[u] = pe * (__uint_as_float(dv[e + u]) - dlt) * dxds;
        }
        pk[e >> 1] = tc_pack2<F16>(ds[0], ds[1]);
      }
      tc::tmem_st16(lane_base + kDSCol + 16 * c, pk);  // dS keys [32 c, 32 c + 32), packed pairs
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    tc::mbar_arrive(ds_ready);

    // ---- thread 0: dQ(t) += dS(t) K(t); then S(t+1), dP(t+1); then the copy of tile t + 2
    if (tid == 0) {
      if (!tc::mbar_wait_spin(ds_ready, t & 1, abort_flag)) {
        ok = false;
      } else {
        tc::fence_after_sync();
        const uint32_t ka = tc::smem_u32(kv_base(t & 1));
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks)
          tc::mma_ts(tbase + kDQCol, tbase + kDSCol + ks * 8, tc::sdesc_sw128(ka + ks * 2048, 16384, 1024), idQ,
                     (t > 0 || ks > 0) ? 1u : 0u);
        tc::mma_commit(q_done);
        if (t + 1 < nkb) {
          if (!tc::mbar_wait_spin(kv_full + ((t + 1) & 1), ((t + 1) >> 1) & 1, abort_flag)) {
            ok = false;
          } else {
            tc::fence_after_sync();
            issue_s(t + 1);
          }
        }
        if (ok && t + 2 < nkb) {
          // tile t's buffer is free once dQ(t) (and everything before it) is done
          if (!tc::mbar_wait_spin(q_done, t & 1, abort_flag)) ok = false;
          else load_kv(t + 2);
        }
      }
      if (!ok) *abort_flag = 1;
    }
  }
  if (!ok && !*abort_flag) *abort_flag = 1;

  // ---- epilogue: dQ rows out of TMEM (zero when no key tile was seen)
  bool have = nkb > 0;
  if (have && !*abort_flag) {
    if (!tc::mbar_wait_spin(q_done, (nkb - 1) & 1, abort_flag)) have = false;
  }
  if (*abort_flag) {
    if (tid == 0) record_error(p, FA_ERR_DEVICE_TIMEOUT, 40);
  } else {
    // warpgroup k stores columns [32 k, 32 k + 32); the TMEM loads are
    // warp-wide (every lane, rows past the sequence too), only rows inside it
    // are stored
    uint16_t* qp = p.dq + (p.cu_q ? 0 : (int64_t)b * p.dq_sb) + ((int64_t)q_row0 + min(i, q_len - 1)) * p.dq_ss +
                   (int64_t)h * p.dq_sh;
    tc::fence_after_sync();
    for (int c = wg; c < D / 32; c += 4) {
      uint32_t v[32];
      if (have) {
        tc::tmem_ld32(lane_base + kDQCol + 32 * c, v);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      if (i < q_len) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w;
          w.x = tc_pack2<F16>(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          w.y = tc_pack2<F16>(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          w.z = tc_pack2<F16>(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
          w.w = tc_pack2<F16>(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
          *reinterpret_cast<uint4*>(qp + 32 * c + e) = w;
        }
      }
    }
  }
  if (*abort_flag && tid == 0) {
    // let the copies and MMAs already issued finish before the CTA leaves
    tc::mma_commit(q_done);
    tc::mbar_wait_drain(q_done, nkb & 1, 100000000ull);
    tc::mbar_wait_drain(kv_full, 0, 100000000ull);
    tc::mbar_wait_drain(kv_full + 1, 0, 100000000ull);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tbase, kTcCols);
}

// ---------------------------------------------------------------------------
// dK, dV: one CTA per (sequence, K/V head, 128-key tile), over every 128-row
// query block of the group's q-heads that can see the tile.  Each block is
// taken in two halves of 64 query rows, h = 0, 1, so that the MMAs of one half
// run while the rows work on the other:
//   S^T_h = K Q_h^T, dP^T_h = V dO_h^T (N = 64) -> P^T_h, dS^T_h (thread
//   (k, r): key r, query columns [16 k, 16 k + 16) of the half) ->
//   dV += P^T_h dO_h, dK += dS^T_h Q_h (K = 64)
// TMEM: S^T_h [64 h, 64 h + 64) then P^T_h over its first 32 columns, dP^T_h
// [128 + 64 h, ...) then dS^T_h over its first 32, dV [256, 256 + D), dK
// [384, 384 + D).  Warps 0-15 are the rows; warp 16 (one thread) issues TMA
// copies and MMAs: dV/dK of half h as soon as its P^T/dS^T are written, then
// S^T/dP^T of half h of the next block once those MMAs are done.  A bounded
// CTA-wide barrier per half separates the reads of S^T_h/dP^T_h from the
// writes over them.  Q/dO blocks in two buffers; LSE and Delta of a block's
// query rows in two shared buffers, filled a block ahead.
// ---------------------------------------------------------------------------
template <int D>
struct DkdvTcCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0, kV = kTile;
  static constexpr int kQO = 2 * kTile;          // [2 buffers][Q, dO]
  static constexpr int kStat = kQO + 4 * kTile;  // [2 buffers][lse2 128, delta 128] floats
  static constexpr int kBar = kStat + 2 * 2 * 128 * 4;
  static constexpr int kUsed = kBar + 256;
  static constexpr int kSmem = (kUsed > 116 * 1024 ? kUsed : 116 * 1024) + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};
constexpr int kDkdvThreads = 544;  // 16 row warps + the issuer warp

template <int D, bool F16>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    dkdv_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using C = DkdvTcCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool issuer_warp = warp == 16;
  const int n_kt = (p.Sk + kTcKeys - 1) / kTcKeys;
  const int kt = (int)(blockIdx.x % n_kt);
  const int64_t r0 = blockIdx.x / n_kt;
  const int g = (int)(r0 % p.Hkv), b = (int)(r0 / p.Hkv);
  const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
  {
    bool bad = q_len < 0 || kv_len < 0 || q_len > p.Sq || kv_len > p.Sk;
    if (p.cu_q) bad |= p.cu_q[b] < 0 || (int64_t)p.cu_q[b + 1] > p.tot_q;
    if (p.cu_k) bad |= p.cu_k[b] < 0 || (int64_t)p.cu_k[b + 1] > p.tot_k;
    if (bad) {
      if (kt == 0 && g == 0 && tid == 0) record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)b);
      return;
    }
  }
  const int k0 = kt * kTcKeys;
  if (k0 >= kv_len) return;
  const int off = kv_len - q_len;
  const int k1 = min(k0 + kTcKeys, kv_len) - 1;
  int ilo = 0, ihi = q_len - 1;
  if (p.causal) ilo = max(ilo, k0 - off);
  if (p.wr >= 0) ilo = max(ilo, k0 - off - p.wr);
  if (p.wl >= 0) ihi = min(ihi, k1 - off + p.wl);
  const int qb0 = ilo > 0 ? ilo / kTcRows : 0;
  const int nqb = ihi >= ilo ? ihi / kTcRows - qb0 + 1 : 0;
  const int n_steps = nqb * p.G;
  const int wg = (warp >> 2) & 3;                              // row threads: query columns [16 wg, +16) of a half
  const int row = 32 * (warp & 3) + (tid & 31), j = k0 + row;  // row threads: this thread's key
  // the pair rules for this key as one interval of query rows [ilo_j, ihi_j]
  int ilo_j = 0, ihi_j = q_len - 1;
  if (j >= kv_len) ihi_j = -1;
  if (p.causal) ilo_j = max(ilo_j, j - off);
  if (p.wr >= 0) ilo_j = max(ilo_j, j - off - p.wr);
  if (p.wl >= 0) ihi_j = min(ihi_j, j - off + p.wl);
  const bool plain = !(p.softcap > 0.f) && !p.alibi;  // logit = scale * s

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* kv_full = bars;        // K and V landed
  uint64_t* qo_full = bars + 1;    // [2] Q/dO buffer landed
  uint64_t* s_done = bars + 3;     // [2 halves] S^T_h and dP^T_h of a block written
  uint64_t* rd_done = bars + 5;    // [2 halves] every row thread has read them (512)
  uint64_t* p_ready = bars + 7;    // [2 halves] P^T_h and dS^T_h written (512)
  uint64_t* m_done = bars + 9;     // [2 halves] dV/dK MMAs of a half (and all before them) done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* stat = reinterpret_cast<float*>(smem + C::kStat);
  if (tid == 0) {
    tc::mbar_init(kv_full, 1);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(qo_full + k, 1);
      tc::mbar_init(s_done + k, 1);
      tc::mbar_init(rd_done + k, 512);
      tc::mbar_init(p_ready + k, 512);
      tc::mbar_init(m_done + k, 1);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTcCols);
    tc::tmem_relinquish();
  }
  const int q_row0 = p.cu_q ? p.cu_q[b] : 0, q_b = p.cu_q ? 0 : b;
  const int k_row0 = p.cu_k ? p.cu_k[b] : 0, k_b = p.cu_k ? 0 : b;
  // LSE (log2 units) and Delta of step s's 128 query rows into buffer s & 1
  auto load_stat = [&](int s) {
    if (tid < 128) {
      const int h = g * p.G + s / nqb;
      const int i = (qb0 + s % nqb) * kTcRows + tid;
      float l2 = 0.f, dl = 0.f;
      if (i < q_len) {
        const int64_t qrow = (int64_t)q_row0 + i;
        l2 = __ldg(p.lse + (p.cu_q ? 0 : (int64_t)b * p.lse_sb) + (int64_t)h * p.lse_sh + qrow * p.lse_ss) * kLog2e;
        dl = p.delta[p.cu_q ? (int64_t)h * p.tot_q + qrow : ((int64_t)b * p.Hq + h) * p.Sq + i];
      }
      stat[(s & 1) * 256 + tid] = l2;
      stat[(s & 1) * 256 + 128 + tid] = dl;
    }
  };
  if (n_steps > 0) load_stat(0);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t lane_base = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
  constexpr uint32_t kDPCol = 128, kDVCol = 256, kDKCol = 384;
  constexpr uint32_t idS = tc::idesc_bf16_f32(128, 64, false, false, F16);
  constexpr uint32_t idO = tc::idesc_bf16_f32(128, D, false, true, F16);
  const uint32_t sK = tc::smem_u32(smem + C::kK), sV = tc::smem_u32(smem + C::kV);
  auto qo_base = [&](int buf) { return smem + C::kQO + buf * 2 * C::kTile; };

  bool ok = true;
  if (issuer_warp) {
    // ------------------------------------------------------------ issuer
    if ((tid & 31) == 0 && n_steps > 0) {
      auto load_qo = [&](int s) {
        unsigned char* dst = qo_base(s & 1);
        const int h = g * p.G + s / nqb;
        const int row_q = q_row0 + (qb0 + s % nqb) * kTcRows;
        tc::mbar_arrive_expect_tx(qo_full + (s & 1), 2 * C::kTile);
        for (int c = 0; c < D / 64; ++c) {
          tc::tma_load_4d(dst + c * 16384, &tq, qo_full + (s & 1), c * 64, h, row_q, q_b);
          tc::tma_load_4d(dst + C::kTile + c * 16384, &tdo, qo_full + (s & 1), c * 64, h, row_q, q_b);
        }
      };
      // S^T_h = K Q_h^T -> [64 h, +64), dP^T_h = V dO_h^T -> [128 + 64 h, +64)
      auto issue_s = [&](int s, int hf) {
        const uint32_t qa = tc::smem_u32(qo_base(s & 1)) + hf * 8192, oa = qa + C::kTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
          tc::mma_ss(tbase + 64 * hf, tc::sdesc_sw128(sK + o, 16, 1024), tc::sdesc_sw128(qa + o, 16, 1024), idS,
                     ks > 0 ? 1u : 0u);
          tc::mma_ss(tbase + kDPCol + 64 * hf, tc::sdesc_sw128(sV + o, 16, 1024), tc::sdesc_sw128(oa + o, 16, 1024),
                     idS, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(s_done + hf);
      };
      tc::tma_prefetch_desc(&tq);
      tc::tma_prefetch_desc(&tdo);
      tc::tma_prefetch_desc(&tk);
      tc::tma_prefetch_desc(&tv);
      tc::mbar_arrive_expect_tx(kv_full, 2 * C::kTile);
      for (int c = 0; c < D / 64; ++c) {
        tc::tma_load_4d(smem + C::kK + c * 16384, &tk, kv_full, c * 64, g, k_row0 + k0, k_b);
        tc::tma_load_4d(smem + C::kV + c * 16384, &tv, kv_full, c * 64, g, k_row0 + k0, k_b);
      }
      load_qo(0);
      if (n_steps > 1) load_qo(1);
      ok = tc::mbar_wait(kv_full, 0, abort_flag) && tc::mbar_wait(qo_full, 0, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0, 0);
        issue_s(0, 1);
      }
      for (int s = 0; ok && s < n_steps; ++s) {
        const uint32_t qa = tc::smem_u32(qo_base(s & 1)), oa = qa + C::kTile;
        for (int hf = 0; ok && hf < 2; ++hf) {
          if (!tc::mbar_wait_spin(p_ready + hf, s & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // dV += P^T_h dO_h, dK += dS^T_h Q_h: K = the half's 64 query rows
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t acc = (s > 0 || hf > 0 || ks > 0) ? 1u : 0u;
            const uint32_t ro = (4 * hf + ks) * 2048;
            tc::mma_ts(tbase + kDVCol, tbase + 64 * hf + ks * 8, tc::sdesc_sw128(oa + ro, 16384, 1024), idO, acc);
            tc::mma_ts(tbase + kDKCol, tbase + kDPCol + 64 * hf + ks * 8, tc::sdesc_sw128(qa + ro, 16384, 1024), idO,
                       acc);
          }
          tc::mma_commit(m_done + hf);
          if (s + 1 < n_steps) {
            // the next block's S^T_h/dP^T_h overwrite P^T_h/dS^T_h: after these MMAs
            if (!tc::mbar_wait_spin(m_done + hf, s & 1, abort_flag) ||
                (hf == 0 && !tc::mbar_wait_spin(qo_full + ((s + 1) & 1), ((s + 1) >> 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            issue_s(s + 1, hf);
          }
        }
        // both halves' dV/dK MMAs are done: this block's Q/dO buffer takes block s + 2
        if (ok && s + 2 < n_steps) load_qo(s + 2);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ rows
    for (int s = 0; s < n_steps; ++s) {
      const int h = g * p.G + s / nqb;
      const int i0 = (qb0 + s % nqb) * kTcRows;
      const float* l2s = stat + (s & 1) * 256;
      const float* dls = l2s + 128;
      const float a_slope = p.alibi ? __ldg(p.alibi + h) * kLog2e : 0.f;
      for (int hf = 0; hf < 2; ++hf) {
        if (!tc::mbar_wait_spin(s_done + hf, s & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        uint32_t sv[16], dv[16];
        tc::tmem_ld16(lane_base + 64 * hf + 16 * wg, sv);
        tc::tmem_ld16(lane_base + kDPCol + 64 * hf + 16 * wg, dv);
        tc::tmem_wait_ld();
        // every row thread has read S^T_h and dP^T_h before any writes over them
        tc::fence_before_sync();
        tc::mbar_arrive(rd_done + hf);
        if (!tc::mbar_wait_spin(rd_done + hf, s & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // every row thread is past block s - 1: its LSE / Delta buffer takes block s + 1's
        if (hf == 0 && s + 1 < n_steps) load_stat(s + 1);
        const int qc = 64 * hf + 16 * wg;  // column of sv[0] within the block
        uint32_t pk[8], dk[8];
        if (plain) {
#pragma unroll
          for (int e4 = 0; e4 < 16; e4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(l2s + qc + e4);
            const float4 d4 = *reinterpret_cast<const float4*>(dls + qc + e4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dl[4] = {d4.x, d4.y, d4.z, d4.w};
            float pv[4], ds[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = i0 + qc + e4 + u;
              const bool in = (i >= ilo_j) & (i <= ihi_j);
              const float pe = in ? fast_exp2(fmaf(__uint_as_float(sv[e4 + u]), p.scale_log2, -lv[u])) : 0.f;
              pv[u] = pe;
              ds[u] = pe * (__uint_as_float(dv[e4 + u]) - dl[u]) * p.scale;
            }
            pk[e4 >> 1] = tc_pack2<F16>(pv[0], pv[1]);
            pk[(e4 >> 1) + 1] = tc_pack2<F16>(pv[2], pv[3]);
            dk[e4 >> 1] = tc_pack2<F16>(ds[0], ds[1]);
            dk[(e4 >> 1) + 1] = tc_pack2<F16>(ds[2], ds[3]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float pv[2], ds[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int q = qc + e + u, i = i0 + q;
              const float sc = __uint_as_float(sv[e + u]);
              float x = -INFINITY, dxds = 0.f;
              if ((i >= ilo_j) & (i <= ihi_j)) {
                if (p.softcap > 0.f) {
                  const float th = tc_softcap_tanh(sc * p.scale, p.inv_softcap);
                  x = th * (p.softcap * kLog2e);
                  dxds = p.scale * (1.f - th * th);
                } else {
                  x = sc * p.scale_log2;
                  dxds = p.scale;
                }
                x -= a_slope * (float)abs(i + off - j);
              }
              const float pe = (x == -INFINITY) ? 0.f : fast_exp2(x - l2s[q]);
              pv[u] = pe;
              ds[u] = pe * (__uint_as_float(dv[e + u]) - dls[q]) * dxds;
            }
            pk[e >> 1] = tc_pack2<F16>(pv[0], pv[1]);
            dk[e >> 1] = tc_pack2<F16>(ds[0], ds[1]);
          }
        }
        tc::tmem_st8(lane_base + 64 * hf + 8 * wg, pk);           // P^T_h, packed pairs
        tc::tmem_st8(lane_base + kDPCol + 64 * hf + 8 * wg, dk);  // dS^T_h
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(p_ready + hf);
      }
      if (!ok) break;
    }
    if (!ok && !*abort_flag) *abort_flag = 1;
  }

  // ---- epilogue (row threads): dK, dV rows out of TMEM (zero when no query block was seen)
  if (!issuer_warp) {
    bool have = n_steps > 0;
    if (have && !*abort_flag) {
      if (!tc::mbar_wait_spin(m_done, (n_steps - 1) & 1, abort_flag) ||
          !tc::mbar_wait_spin(m_done + 1, (n_steps - 1) & 1, abort_flag))
        have = false;
    }
    if (*abort_flag) {
      if (tid == 0) record_error(p, FA_ERR_DEVICE_TIMEOUT, 41);
    } else {
      const int jc = min(j, kv_len - 1);
      uint16_t* kp = p.dk + (p.cu_k ? 0 : (int64_t)b * p.dk_sb) + ((int64_t)k_row0 + jc) * p.dk_ss + (int64_t)g * p.dk_sh;
      uint16_t* vp = p.dv + (p.cu_k ? 0 : (int64_t)b * p.dv_sb) + ((int64_t)k_row0 + jc) * p.dv_ss + (int64_t)g * p.dv_sh;
      tc::fence_after_sync();
      // warpgroup k: chunks k, k + 4, ... of [dV chunks | dK chunks]
      for (int c = wg; c < 2 * (D / 32); c += 4) {
        const bool is_k = c >= D / 32;
        const int cc = is_k ? c - D / 32 : c;
        uint32_t v[32];
        if (have) {
          tc::tmem_ld32(lane_base + (is_k ? kDKCol : kDVCol) + 32 * cc, v);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (j < kv_len) {
          uint16_t* dst = (is_k ? kp : vp) + 32 * cc;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = tc_pack2<F16>(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            w.y = tc_pack2<F16>(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            w.z = tc_pack2<F16>(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
            w.w = tc_pack2<F16>(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
            *reinterpret_cast<uint4*>(dst + e) = w;
          }
        }
      }
    }
  } else if (*abort_flag && (tid & 31) == 0) {
    // let the copies and MMAs already issued finish before the CTA leaves
    tc::mma_commit(m_done);
    tc::mbar_wait_drain(m_done, n_steps & 1, 100000000ull);
    tc::mbar_wait_drain(kv_full, 0, 100000000ull);
    tc::mbar_wait_drain(qo_full, 0, 100000000ull);
    tc::mbar_wait_drain(qo_full + 1, 0, 100000000ull);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tbase, kTcCols);
}

bool encode_tile(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int batch, int64_t s_h,
                 int64_t s_row, int64_t s_b, bool f16) {
  return encode_4d_bf16(m, base, d, heads, rows, batch, s_h, s_row, s_b, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, f16);
}

template <int D, bool F16>
cudaError_t launch_bwd_tc_d(const Params& p, cudaStream_t st, bool* launched) {
  *launched = false;
  const bool vq = p.cu_q != nullptr, vk = p.cu_k != nullptr;
  const int64_t q_rows = vq ? p.tot_q : p.Sq, k_rows = vk ? p.tot_k : p.Sk;
  const int qb = vq ? 1 : p.n_seq, kb = vk ? 1 : p.n_seq;
  auto sb = [](int nb, int64_t s_b, int64_t s_row) { return (nb == 1 || s_b == 0) ? s_row : s_b; };
  CUtensorMap mq, mdo, mk, mv;
  if (q_rows <= 0 || k_rows <= 0) return cudaSuccess;
  if (!encode_tile(&mq, p.q, D, p.Hq, q_rows, qb, p.q_sh, p.q_ss, sb(qb, p.q_sb, p.q_ss), F16) ||
      !encode_tile(&mdo, p.dout, D, p.Hq, q_rows, qb, p.do_sh, p.do_ss, sb(qb, p.do_sb, p.do_ss), F16) ||
      !encode_tile(&mk, p.k, D, p.Hkv, k_rows, kb, p.k_sh, p.k_ss, sb(kb, p.k_sb, p.k_ss), F16) ||
      !encode_tile(&mv, p.v, D, p.Hkv, k_rows, kb, p.v_sh, p.v_ss, sb(kb, p.v_sb, p.v_ss), F16))
    return cudaSuccess;  // layout without tensor maps: the caller takes the warp-level kernel
  cudaError_t e = ensure_smem_attr<dq_tc_kernel<D, F16>>(DqTcCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_attr<dkdv_tc_kernel<D, F16>>(DkdvTcCfg<D>::kSmem)) != cudaSuccess) return e;
  const int64_t n_kt = (p.Sk + kTcKeys - 1) / kTcKeys;
  const int64_t g1 = (int64_t)p.n_seq * p.Hkv * n_kt;
  if (g1 > 0) dkdv_tc_kernel<D, F16><<<(unsigned)g1, kDkdvThreads, DkdvTcCfg<D>::kSmem, st>>>(p, mq, mdo, mk, mv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n_qt = (p.Sq + kTcRows - 1) / kTcRows;
  const int64_t grid = (int64_t)p.n_seq * p.Hq * n_qt;
  if (grid > 0) dq_tc_kernel<D, F16><<<(unsigned)grid, 512, DqTcCfg<D>::kSmem, st>>>(p, mq, mdo, mk, mv);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace

// dK/dV and dQ on tcgen05; *launched = false (nothing enqueued) when a tensor
// map cannot describe the layout.
cudaError_t launch_bwd_tc(const Params& p, cudaStream_t st, bool* launched) {
  if (p.f16) return p.d == 64 ? launch_bwd_tc_d<64, true>(p, st, launched) : launch_bwd_tc_d<128, true>(p, st, launched);
  return p.d == 64 ? launch_bwd_tc_d<64, false>(p, st, launched) : launch_bwd_tc_d<128, false>(p, st, launched);
}

}  // namespace mfa
