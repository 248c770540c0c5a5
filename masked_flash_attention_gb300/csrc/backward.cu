// backward.cu -- gradients dQ, dK, dV of the masked attention forward
// (InfiniTrain pull request 193, "FlashAttention native backend": the
// FlashAttention-2 causal forward and backward kernels; "Framework 与
// autograd": the autograd function around them).
//
// Per (sequence, q-head h, K/V head g): with P recomputed from the forward's
// LSE (P = exp(x - LSE), x the final logit), Delta = rowsum(dO * O),
// dP = dO V^T, dS = P * (dP - Delta) * dx/ds (dx/ds = scale, or
// scale * (1 - tanh^2) under the soft-cap):
//   dV_g = sum_h P^T dO_h,   dK_g = sum_h dS^T Q_h,   dQ_h = dS K_g.
// Three kernels, no atomics (the result does not depend on scheduling):
//   delta_kernel  Delta per (row, q-head)
//   dkdv_kernel   one CTA per (sequence, K/V head, 64-key tile); each warp
//                 owns 16 keys (mma M side) and accumulates its dK and dV rows
//                 over every 16-row query block of the group's q-heads that can
//                 see the tile, so the grouped-query sum happens in registers
//   dq_kernel     one CTA per (sequence, q-head, 64-row tile); each warp owns
//                 16 query rows (M side) and accumulates dQ over the key tiles
//                 its rows can see
// S and dP are computed in both kernels.  The pair rules, the soft-cap and
// ALiBi are the forward's; a row with no allowed key has LSE = -inf and gets
// P = 0.  Rows and keys past a sequence are read clamped (finite) and masked.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "host_util.h"
#include "mma_sync.cuh"

namespace mfa {

namespace {

constexpr int kBwdWarps = 4;
constexpr int kBwdThreads = 32 * kBwdWarps;
constexpr int kKeyTile = 64;  // keys per dK/dV CTA (16 per warp)
constexpr int kRowTile = 64;  // query rows per dQ CTA (16 per warp)
constexpr int kBlk = 16;      // query rows per dK/dV step

// tanh(x / cap) by the identity of the forward's soft-cap.
__device__ __forceinline__ float softcap_tanh(float x, float inv_cap) {
  const float y = x * inv_cap;
  const float t = fast_exp2(-2.f * kLog2e * fabsf(y));
  return copysignf(__fdividef(1.f - t, 1.f + t), y);
}

// Logit of one raw dot product s in log2 units (-inf when the pair is dropped
// or the row is past the sequence) and its derivative dx/ds in natural units.
__device__ __forceinline__ float bwd_logit(const Params& p, float s, int h, int i, int j, int off, int kv_len,
                                           int q_len, float& dxds) {
  if (i >= q_len || !pair_allowed(p, i, j, off, kv_len)) {
    dxds = 0.f;
    return -INFINITY;
  }
  float x;
  if (p.softcap > 0.f) {
    const float t = softcap_tanh(s * p.scale, p.inv_softcap);
    x = t * (p.softcap * kLog2e);
    dxds = p.scale * (1.f - t * t);
  } else {
    x = s * p.scale_log2;
    dxds = p.scale;
  }
  if (p.alibi) x -= __ldg(p.alibi + h) * kLog2e * (float)abs(i + off - j);
  return x;
}

// Sequence lengths, checked against the planned sizes (the lengths come from
// device memory); false (error recorded once per sequence) when they do not fit.
__device__ __forceinline__ bool bwd_lengths(const Params& p, int b, bool report, int& q_len, int& kv_len) {
  q_len = seq_qlen(p, b);
  kv_len = seq_klen(p, b);
  bool bad = q_len < 0 || kv_len < 0 || q_len > p.Sq || kv_len > p.Sk;
  if (p.cu_q) bad |= p.cu_q[b] < 0 || (int64_t)p.cu_q[b + 1] > p.tot_q;
  if (p.cu_k) bad |= p.cu_k[b] < 0 || (int64_t)p.cu_k[b + 1] > p.tot_k;
  if (bad && report) record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)b);
  return !bad;
}

// element offset of query-side row i (q-head h) of sequence b for a tensor
// with strides (sb, ss, sh) laid out like q
__device__ __forceinline__ int64_t qside(const Params& p, int64_t sb, int64_t ss, int64_t sh, int b, int h, int i) {
  const int64_t row = p.cu_q ? (int64_t)p.cu_q[b] + i : (int64_t)i;
  return (p.cu_q ? 0 : (int64_t)b * sb) + row * ss + (int64_t)h * sh;
}
// ... and of key row j (K/V head g) for a tensor laid out like k
__device__ __forceinline__ int64_t kside(const Params& p, int64_t sb, int64_t ss, int64_t sh, int b, int g, int j) {
  const int64_t row = p.cu_k ? (int64_t)p.cu_k[b] + j : (int64_t)j;
  return (p.cu_k ? 0 : (int64_t)b * sb) + row * ss + (int64_t)g * sh;
}
// index of (sequence b, q-head h, row i) in the Delta buffer (the LSE layout:
// [B, Hq, Sq], or [Hq, total_q] for packed sequences)
__device__ __forceinline__ int64_t delta_index(const Params& p, int b, int h, int i) {
  return p.cu_q ? (int64_t)h * p.tot_q + p.cu_q[b] + i : ((int64_t)b * p.Hq + h) * p.Sq + i;
}
__device__ __forceinline__ float lse_log2(const Params& p, int b, int h, int i) {
  const int64_t row = p.cu_q ? (int64_t)p.cu_q[b] + i : (int64_t)i;
  return __ldg(p.lse + (p.cu_q ? 0 : (int64_t)b * p.lse_sb) + (int64_t)h * p.lse_sh + row * p.lse_ss) * kLog2e;
}

template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (F16) return __half22float2(*reinterpret_cast<const __half2*>(&v));
  else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// ---------------------------------------------------------------------------
// Delta = rowsum(dO * O), one warp per (row, q-head)
// ---------------------------------------------------------------------------
template <int D, bool F16>
__global__ void __launch_bounds__(256) delta_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t rows = p.cu_q ? p.tot_q : (int64_t)p.n_seq * p.Sq;
  if (w >= rows * p.Hq) return;
  const int h = (int)(w % p.Hq);
  const int64_t t = w / p.Hq;
  int64_t oo, od, di;
  if (p.cu_q) {  // packed row t
    oo = t * p.o_ss + (int64_t)h * p.o_sh;
    od = t * p.do_ss + (int64_t)h * p.do_sh;
    di = (int64_t)h * p.tot_q + t;
  } else {
    const int64_t b = t / p.Sq, i = t % p.Sq;
    oo = b * p.o_sb + i * p.o_ss + (int64_t)h * p.o_sh;
    od = b * p.do_sb + i * p.do_ss + (int64_t)h * p.do_sh;
    di = (b * p.Hq + h) * p.Sq + i;
  }
  constexpr int kPer = D / 32;  // elements per lane
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < kPer; c += 2) {
    const uint32_t a = *reinterpret_cast<const uint32_t*>(p.o + oo + lane * kPer + c);
    const uint32_t g = *reinterpret_cast<const uint32_t*>(p.dout + od + lane * kPer + c);
    const float2 fa = unpack2<F16>(a), fg = unpack2<F16>(g);
    acc += fa.x * fg.x + fa.y * fg.y;
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) p.delta[di] = acc;
}

// ---------------------------------------------------------------------------
// dK, dV
// ---------------------------------------------------------------------------
template <int D>
struct DkdvSmem {
  static constexpr int kTile = kKeyTile * D * 2;  // K or V tile
  static constexpr int kBlkBytes = kBlk * D * 2;  // Q or dO block
  static constexpr int kK = 0, kV = kTile;
  static constexpr int kQ = 2 * kTile;                   // [2 buffers]
  static constexpr int kDO = kQ + 2 * kBlkBytes;         // [2 buffers]
  static constexpr int kStat = kDO + 2 * kBlkBytes;      // [2 buffers][lse2 16, delta 16]
  static constexpr int kTotal = kStat + 2 * 2 * kBlk * 4;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kBwdThreads) dkdv_kernel(const Params p) {
  using S = DkdvSmem<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_kt = (p.Sk + kKeyTile - 1) / kKeyTile;
  const int kt = (int)(blockIdx.x % n_kt);
  const int64_t r = blockIdx.x / n_kt;
  const int g = (int)(r % p.Hkv), b = (int)(r / p.Hkv);
  int q_len, kv_len;
  if (!bwd_lengths(p, b, kt == 0 && g == 0 && tid == 0, q_len, kv_len)) return;
  const int k0 = kt * kKeyTile;
  if (k0 >= kv_len) return;
  const int off = kv_len - q_len;
  // query rows that can see a key of [k0, k0 + 63] under the pair rules
  const int k1 = min(k0 + kKeyTile, kv_len) - 1;
  int ilo = 0, ihi = q_len - 1;
  if (p.causal) ilo = max(ilo, k0 - off);
  if (p.wr >= 0) ilo = max(ilo, k0 - off - p.wr);
  if (p.wl >= 0) ihi = min(ihi, k1 - off + p.wl);
  const int qb0 = ilo > 0 ? ilo / kBlk : 0;
  const int nqb = ihi >= ilo ? ihi / kBlk - qb0 + 1 : 0;
  const int n_steps = nqb * p.G;
  const uint32_t sb = (uint32_t)__cvta_generic_to_shared(smem);
  constexpr int kC = D / 8;  // 16-byte chunks per row

  // K and V tile (rows past the sequence read its last key: finite, masked)
  for (int idx = tid; idx < kKeyTile * kC; idx += kBwdThreads) {
    const int rr = idx / kC, c = idx % kC;
    const int j = min(k0 + rr, kv_len - 1);
    cp_async16(sb + S::kK + swz<D>(rr, c), p.k + kside(p, p.k_sb, p.k_ss, p.k_sh, b, g, j) + c * 8);
    cp_async16(sb + S::kV + swz<D>(rr, c), p.v + kside(p, p.v_sb, p.v_ss, p.v_sh, b, g, j) + c * 8);
  }
  float* stat = reinterpret_cast<float*>(smem + S::kStat);
  auto load_step = [&](int s, int buf) {
    const int h = g * p.G + s / nqb;
    const int i0 = (qb0 + s % nqb) * kBlk;
    for (int idx = tid; idx < kBlk * kC; idx += kBwdThreads) {
      const int rr = idx / kC, c = idx % kC;
      const int i = min(i0 + rr, q_len - 1);
      cp_async16(sb + S::kQ + buf * S::kBlkBytes + swz<D>(rr, c), p.q + qside(p, p.q_sb, p.q_ss, p.q_sh, b, h, i) + c * 8);
      cp_async16(sb + S::kDO + buf * S::kBlkBytes + swz<D>(rr, c),
                 p.dout + qside(p, p.do_sb, p.do_ss, p.do_sh, b, h, i) + c * 8);
    }
    if (tid < kBlk) {
      const int i = min(i0 + tid, q_len - 1);
      stat[buf * 2 * kBlk + tid] = lse_log2(p, b, h, i);
      stat[buf * 2 * kBlk + kBlk + tid] = p.delta[delta_index(p, b, h, i)];
    }
  };
  if (n_steps > 0) load_step(0, 0);
  cp_async_commit();

  const int g8 = lane >> 2, c4 = lane & 3, mi = lane >> 3;
  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;

  for (int s = 0; s < n_steps; ++s) {
    const int buf = s & 1;
    cp_async_wait<0>();
    __syncthreads();  // this step's block (and the K/V tile) landed; the other buffer is free
    if (s + 1 < n_steps) load_step(s + 1, buf ^ 1);
    cp_async_commit();
    const int h = g * p.G + s / nqb;
    const int i0 = (qb0 + s % nqb) * kBlk;
    const uint32_t sQ = sb + S::kQ + buf * S::kBlkBytes, sO = sb + S::kDO + buf * S::kBlkBytes;
    const float* lse2 = stat + buf * 2 * kBlk;
    const float* dlt = lse2 + kBlk;

    // S^T and dP^T: [16 keys x 16 rows] as two n-blocks of 8 rows
    float st[2][4], dpt[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[nb][e] = dpt[nb][e] = 0.f;
    // (the four accumulators take turns, so no MMA waits on the one before it)
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      uint32_t ka[2][4], va[2][4], qf[2][4], of[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int kr = 16 * warp + (lane & 7) + 8 * (mi & 1), kc = 2 * (ks + u) + (mi >> 1);
        ldsm_x4(sb + S::kK + swz<D>(kr, kc), ka[u][0], ka[u][1], ka[u][2], ka[u][3]);
        ldsm_x4(sb + S::kV + swz<D>(kr, kc), va[u][0], va[u][1], va[u][2], va[u][3]);
      }
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        ldsm_x4(sQ + swz<D>(8 * nb + (lane & 7), 2 * ks + mi), qf[nb][0], qf[nb][1], qf[nb][2], qf[nb][3]);
        ldsm_x4(sO + swz<D>(8 * nb + (lane & 7), 2 * ks + mi), of[nb][0], of[nb][1], of[nb][2], of[nb][3]);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          mma_bf16<F16>(st[nb], ka[u], qf[nb][2 * u], qf[nb][2 * u + 1]);
          mma_bf16<F16>(dpt[nb], va[u], of[nb][2 * u], of[nb][2 * u + 1]);
        }
    }
    // P^T and dS^T; element e of n-block nb: key 16 warp + g8 + 8 (e >> 1), row 8 nb + 2 c4 + (e & 1)
    uint32_t pa[4], da[4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      float pv[4], dsv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = 8 * nb + 2 * c4 + (e & 1);
        const int j = k0 + 16 * warp + g8 + 8 * (e >> 1);
        float dxds;
        const float x = bwd_logit(p, st[nb][e], h, i0 + rr, j, off, kv_len, q_len, dxds);
        const float pe = (x == -INFINITY) ? 0.f : fast_exp2(x - lse2[rr]);
        pv[e] = pe;
        dsv[e] = pe * (dpt[nb][e] - dlt[rr]) * dxds;
      }
      // C fragments of the two n-blocks are the A fragment of a 16x16 operand
      pa[2 * nb] = pack_bf16<F16>(pv[0], pv[1]);
      pa[2 * nb + 1] = pack_bf16<F16>(pv[2], pv[3]);
      da[2 * nb] = pack_bf16<F16>(dsv[0], dsv[1]);
      da[2 * nb + 1] = pack_bf16<F16>(dsv[2], dsv[3]);
    }
    const uint32_t pA[4] = {pa[0], pa[1], pa[2], pa[3]};
    const uint32_t dA[4] = {da[0], da[1], da[2], da[3]};
    // dV += P^T dO, dK += dS^T Q: B = [16 rows x 8 d] per n-block, by transposed loads
    // (the next n-pair's B fragments are loaded before this pair's MMAs)
    const int rrt = (lane & 7) + 8 * ((lane >> 3) & 1);
    uint32_t ob[2][4], qb[2][4];
    ldsm_x4_t(sO + swz<D>(rrt, lane >> 4), ob[0][0], ob[0][1], ob[0][2], ob[0][3]);
    ldsm_x4_t(sQ + swz<D>(rrt, lane >> 4), qb[0][0], qb[0][1], qb[0][2], qb[0][3]);
#pragma unroll
    for (int np = 0; np < D / 16; ++np) {
      const int cur = np & 1;
      if (np + 1 < D / 16) {
        const int cc = 2 * (np + 1) + (lane >> 4);
        ldsm_x4_t(sO + swz<D>(rrt, cc), ob[cur ^ 1][0], ob[cur ^ 1][1], ob[cur ^ 1][2], ob[cur ^ 1][3]);
        ldsm_x4_t(sQ + swz<D>(rrt, cc), qb[cur ^ 1][0], qb[cur ^ 1][1], qb[cur ^ 1][2], qb[cur ^ 1][3]);
      }
      mma_bf16<F16>(dv[2 * np], pA, ob[cur][0], ob[cur][1]);
      mma_bf16<F16>(dk[2 * np], dA, qb[cur][0], qb[cur][1]);
      mma_bf16<F16>(dv[2 * np + 1], pA, ob[cur][2], ob[cur][3]);
      mma_bf16<F16>(dk[2 * np + 1], dA, qb[cur][2], qb[cur][3]);
    }
  }
  cp_async_wait<0>();
  // rows: key 16 warp + g8 (+ 8); columns: d 8 n + 2 c4 (+ 1)
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = k0 + 16 * warp + g8 + 8 * hh;
    if (j >= kv_len) continue;
    uint16_t* kp = p.dk + kside(p, p.dk_sb, p.dk_ss, p.dk_sh, b, g, j);
    uint16_t* vp = p.dv + kside(p, p.dv_sb, p.dv_ss, p.dv_sh, b, g, j);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<uint32_t*>(kp + 8 * n + 2 * c4) = pack_bf16<F16>(dk[n][2 * hh], dk[n][2 * hh + 1]);
      *reinterpret_cast<uint32_t*>(vp + 8 * n + 2 * c4) = pack_bf16<F16>(dv[n][2 * hh], dv[n][2 * hh + 1]);
    }
  }
}

// ---------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------
template <int D>
struct DqSmem {
  static constexpr int kRows = kRowTile * D * 2;  // Q or dO tile, K or V tile
  static constexpr int kQ = 0, kDO = kRows;
  static constexpr int kKV = 2 * kRows;           // [2 buffers][K, V]
  static constexpr int kTotal = kKV + 2 * 2 * kRows;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kBwdThreads) dq_kernel(const Params p) {
  using S = DqSmem<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_qt = (p.Sq + kRowTile - 1) / kRowTile;
  const int qt = (int)(blockIdx.x % n_qt);
  const int64_t r = blockIdx.x / n_qt;
  const int h = (int)(r % p.Hq), b = (int)(r / p.Hq);
  const int g = h / p.G;
  int q_len, kv_len;
  if (!bwd_lengths(p, b, false, q_len, kv_len)) return;
  const int i0 = qt * kRowTile;
  if (i0 >= q_len) return;
  const int off = kv_len - q_len;
  int jlo, jhi;
  key_range(p, i0, min(i0 + kRowTile, q_len) - 1, off, kv_len, jlo, jhi);
  const int kb0 = jlo > 0 ? jlo / kRowTile : 0;
  const int nkb = jhi >= jlo ? jhi / kRowTile - kb0 + 1 : 0;
  const uint32_t sb = (uint32_t)__cvta_generic_to_shared(smem);
  constexpr int kC = D / 8;

  for (int idx = tid; idx < kRowTile * kC; idx += kBwdThreads) {
    const int rr = idx / kC, c = idx % kC;
    const int i = min(i0 + rr, q_len - 1);
    cp_async16(sb + S::kQ + swz<D>(rr, c), p.q + qside(p, p.q_sb, p.q_ss, p.q_sh, b, h, i) + c * 8);
    cp_async16(sb + S::kDO + swz<D>(rr, c), p.dout + qside(p, p.do_sb, p.do_ss, p.do_sh, b, h, i) + c * 8);
  }
  cp_async_commit();
  auto load_tile = [&](int t, int buf) {
    const int j0 = (kb0 + t) * kRowTile;
    const uint32_t base = sb + S::kKV + buf * 2 * S::kRows;
    for (int idx = tid; idx < kRowTile * kC; idx += kBwdThreads) {
      const int rr = idx / kC, c = idx % kC;
      const int j = min(j0 + rr, kv_len - 1);
      cp_async16(base + swz<D>(rr, c), p.k + kside(p, p.k_sb, p.k_ss, p.k_sh, b, g, j) + c * 8);
      cp_async16(base + S::kRows + swz<D>(rr, c), p.v + kside(p, p.v_sb, p.v_ss, p.v_sh, b, g, j) + c * 8);
    }
  };
  if (nkb > 0) load_tile(0, 0);
  cp_async_commit();

  const int g8 = lane >> 2, c4 = lane & 3, mi = lane >> 3;
  // this warp's rows: i0 + 16 warp + g8 (+ 8)
  const int ir0 = i0 + 16 * warp + g8, ir1 = ir0 + 8;
  const float lse0 = ir0 < q_len ? lse_log2(p, b, h, ir0) : 0.f;
  const float lse1 = ir1 < q_len ? lse_log2(p, b, h, ir1) : 0.f;
  const float dl0 = ir0 < q_len ? p.delta[delta_index(p, b, h, ir0)] : 0.f;
  const float dl1 = ir1 < q_len ? p.delta[delta_index(p, b, h, ir1)] : 0.f;

  cp_async_wait<1>();
  __syncthreads();
  // Q and dO of this warp's 16 rows as A fragments, kept in registers
  uint32_t qa[D / 16][4], oa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int rr = 16 * warp + (lane & 7) + 8 * (mi & 1), cc = 2 * ks + (mi >> 1);
    ldsm_x4(sb + S::kQ + swz<D>(rr, cc), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    ldsm_x4(sb + S::kDO + swz<D>(rr, cc), oa[ks][0], oa[ks][1], oa[ks][2], oa[ks][3]);
  }
  float dq[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;

  for (int t = 0; t < nkb; ++t) {
    const int buf = t & 1;
    cp_async_wait<0>();
    __syncthreads();
    if (t + 1 < nkb) load_tile(t + 1, buf ^ 1);
    cp_async_commit();
    const int j0 = (kb0 + t) * kRowTile;
    const uint32_t sK = sb + S::kKV + buf * 2 * S::kRows, sV = sK + S::kRows;
#pragma unroll 1
    for (int sk = 0; sk < kRowTile / 16; ++sk) {
      // S and dP: [16 rows x 16 keys] as two n-blocks of 8 keys
      float sa[2][4], dp[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nb][e] = dp[nb][e] = 0.f;
      // (the four accumulators take turns, so no MMA waits on the one before it)
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t kf[2][4], vf[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const int kr = 16 * sk + 8 * nb + (lane & 7);
          ldsm_x4(sK + swz<D>(kr, 2 * ks + mi), kf[nb][0], kf[nb][1], kf[nb][2], kf[nb][3]);
          ldsm_x4(sV + swz<D>(kr, 2 * ks + mi), vf[nb][0], vf[nb][1], vf[nb][2], vf[nb][3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            mma_bf16<F16>(sa[nb], qa[ks + u], kf[nb][2 * u], kf[nb][2 * u + 1]);
            mma_bf16<F16>(dp[nb], oa[ks + u], vf[nb][2 * u], vf[nb][2 * u + 1]);
          }
      }
      // dS; element e of n-block nb: row g8 + 8 (e >> 1), key 8 nb + 2 c4 + (e & 1)
      uint32_t da[4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        float dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = (e >> 1) ? ir1 : ir0;
          const int j = j0 + 16 * sk + 8 * nb + 2 * c4 + (e & 1);
          float dxds;
          const float x = bwd_logit(p, sa[nb][e], h, i, j, off, kv_len, q_len, dxds);
          const float pe = (x == -INFINITY) ? 0.f : fast_exp2(x - ((e >> 1) ? lse1 : lse0));
          dsv[e] = pe * (dp[nb][e] - ((e >> 1) ? dl1 : dl0)) * dxds;
        }
        da[2 * nb] = pack_bf16<F16>(dsv[0], dsv[1]);
        da[2 * nb + 1] = pack_bf16<F16>(dsv[2], dsv[3]);
      }
      const uint32_t dA[4] = {da[0], da[1], da[2], da[3]};
      // dQ += dS K: B = [16 keys x 8 d] per n-block, by transposed loads of K rows
      const int rrt = 16 * sk + (lane & 7) + 8 * ((lane >> 3) & 1);
      uint32_t kb[2][4];
      ldsm_x4_t(sK + swz<D>(rrt, lane >> 4), kb[0][0], kb[0][1], kb[0][2], kb[0][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int cur = np & 1;
        if (np + 1 < D / 16)
          ldsm_x4_t(sK + swz<D>(rrt, 2 * (np + 1) + (lane >> 4)), kb[cur ^ 1][0], kb[cur ^ 1][1], kb[cur ^ 1][2],
                    kb[cur ^ 1][3]);
        mma_bf16<F16>(dq[2 * np], dA, kb[cur][0], kb[cur][1]);
        mma_bf16<F16>(dq[2 * np + 1], dA, kb[cur][2], kb[cur][3]);
      }
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int i = hh ? ir1 : ir0;
    if (i >= q_len) continue;
    uint16_t* qp = p.dq + qside(p, p.dq_sb, p.dq_ss, p.dq_sh, b, h, i);
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<uint32_t*>(qp + 8 * n + 2 * c4) = pack_bf16<F16>(dq[n][2 * hh], dq[n][2 * hh + 1]);
  }
}

template <int D, bool F16>
cudaError_t launch_bwd_d(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  cudaError_t e;
  if ((e = ensure_smem_attr<dkdv_kernel<D, F16>>(DkdvSmem<D>::kTotal)) != cudaSuccess) return e;
  if ((e = ensure_smem_attr<dq_kernel<D, F16>>(DqSmem<D>::kTotal)) != cudaSuccess) return e;
  if (ev_begin && (e = cudaEventRecord(ev_begin, st)) != cudaSuccess) return e;
  const int64_t rows = p.cu_q ? p.tot_q : (int64_t)p.n_seq * p.Sq;
  const int64_t warps = rows * p.Hq;
  if (warps > 0) delta_kernel<D, F16><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // dK/dV and dQ on the tensor cores when tensor maps describe the layout,
  // else the warp-level kernels below
  bool tc = false;
  if ((e = launch_bwd_tc(p, st, &tc)) != cudaSuccess || tc) return e;
  const int64_t n_kt = (p.Sk + kKeyTile - 1) / kKeyTile, n_qt = (p.Sq + kRowTile - 1) / kRowTile;
  const int64_t g1 = (int64_t)p.n_seq * p.Hkv * n_kt, g2 = (int64_t)p.n_seq * p.Hq * n_qt;
  if (g1 > 0) dkdv_kernel<D, F16><<<(unsigned)g1, kBwdThreads, DkdvSmem<D>::kTotal, st>>>(p);
  if (g2 > 0) dq_kernel<D, F16><<<(unsigned)g2, kBwdThreads, DqSmem<D>::kTotal, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  if (p.f16) return p.d == 64 ? launch_bwd_d<64, true>(p, st, ev_begin) : launch_bwd_d<128, true>(p, st, ev_begin);
  return p.d == 64 ? launch_bwd_d<64, false>(p, st, ev_begin) : launch_bwd_d<128, false>(p, st, ev_begin);
}

}  // namespace mfa
