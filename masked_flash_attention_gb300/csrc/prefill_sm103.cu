// prefill_sm103.cu -- masked flash-attention forward for many query rows on
// the 5th-generation tensor cores of sm_103a (tcgen05 + TMEM + TMA).
//
// The method is the tiled, online-softmax attention of the ExecuTorch pull
// request 10466 "Summary": q@k is cut into chunks along both the query and the
// key dimension, the softmax is accumulated progressively and rescaled at the
// end; an all -inf chunk must not poison the running values.  Chunks whose
// every pair is masked are not computed at all: the scheduler (sched.cu) left
// them out of each item's key-tile list.
//
// CTA = two 128-row query sub-tiles that read the same K/V head: two q-heads
// of one grouped-query group (InfiniTrain pull request 193 "Transformer 接入":
// the kernel shares the K/V heads instead of expanding them) or, with one
// q-head per K/V head, two consecutive row tiles.  Every K/V tile is loaded
// once by TMA for both.  The two key-tile lists are merged; a sub-tile skips
// the tiles that are not on its own list.
//
// Warp roles (12 warps = 3 warpgroups):
//   warp 0      TMA producer: Q once, then K tiles through an NS-stage ring
//   warp 1      MMA issuer for sub-tile 0 (one thread) and TMEM owner
//   warp 2      TMA producer: V tiles through an NS-stage ring
//   warp 3      MMA issuer for sub-tile 1 (one thread)
//   warps 4..7  softmax warpgroup for sub-tile 0, warps 8..11 for sub-tile 1
// Registers: the block launches with 168 per thread (3 warps share an SM
// sub-partition); warpgroup 0 (producer, MMA) hands registers back with
// setmaxnreg and the softmax warpgroups take 216, enough to keep a whole
// 128-key row of S in registers for one pass: max, exponentiate, sum, store P.
// The kernel is specialised on the additive term (none, dense, top-k) and on
// the soft-cap; a PARTIAL tile applies the pair rules as one column range per
// row, and top-k tiles stage their keys' expiry rows and bias in smem.
// TMEM (512 columns): S_t = Q_t K^T in columns [128 t, 128 t + 128), fp32;
// P_t (bf16, two per column) overwrites the first 64 of them; O_t in
// [256 + D t, 256 + D t + D).  Per key tile j the two MMA issuers put out
//   PV_0(j-1), QK_0(j) | PV_1(j-1), QK_1(j)
// in that order, so that sub-tile 0's softmax of tile j overlaps sub-tile 1's
// MMAs and vice versa.  Each softmax thread owns one query row (32x32b TMEM loads), so the
// row max and row sum need no cross-lane reduction.  The running max is the
// exponent reference and is only raised when the row max exceeds it by more
// than 2^8 (in log2 units), so O in TMEM is rarely rescaled.  A fully masked
// row keeps reference -inf, exponentiates against 0, and ends with l = 0:
// O = 0, LSE = -inf.
//
// Every mbarrier wait is bounded (1 s); on a time-out the kernel records
// FA_ERR_DEVICE_TIMEOUT in the workspace error word, every role stops, in-flight
// MMAs are drained and TMEM is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <mutex>
#include <type_traits>

#include "fa_device.cuh"
#include "host_util.h"
#include "tc_sm103.cuh"

namespace mfa {

namespace {

constexpr int kPrefillThreads = 384;
// Register split (setmaxnreg): the kernel is built to launch with exactly
// kLaunchRegs per thread; warpgroup 0 (producer, MMA) gives registers back and
// the two softmax warpgroups take them, so that a 128-key row of S fits.
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 72;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kProducerRegs + 256 * kSoftmaxRegs <= kPrefillThreads * kLaunchRegs,
              "the register split must fit the block's launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct PCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;          // K/V stages
  static constexpr int kTileBytes = 128 * D * 2;          // one 128-row bf16 tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + NS * kTileBytes;
  static constexpr int kBarOff = kVOff + NS * kTileBytes;
  static constexpr int kSmem = kBarOff + 256 + 4096 + 1024;  // barriers, top-k staging, alignment slack
  static constexpr uint32_t kOCol = 256;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct SubTile {
  bool valid;   // sequence passed the scheduler's checks and the sub-tile exists
  int h, rt, count;
  const int32_t* tiles;
};

// Merged walk over two ascending key-tile lists.
struct Merge {
  const int32_t* l0;
  const int32_t* l1;
  int c0, c1, i0, i1;
  __device__ __forceinline__ void init(const SubTile (&st)[2]) {
    l0 = st[0].tiles; l1 = st[1].tiles;
    c0 = st[0].valid ? st[0].count : 0;
    c1 = st[1].valid ? st[1].count : 0;
    i0 = i1 = 0;
  }
  __device__ __forceinline__ bool next(int& kt, bool& in0, bool& in1, bool& part0, bool& part1) {
    int e0 = i0 < c0 ? __ldg(l0 + i0) : 0x7ffffffe;
    int e1 = i1 < c1 ? __ldg(l1 + i1) : 0x7ffffffe;
    int k0 = e0 >> 1, k1 = e1 >> 1;
    kt = min(k0, k1);
    if (kt >= 0x3fffffff) return false;
    in0 = (k0 == kt); in1 = (k1 == kt);
    part0 = in0 && (e0 & 1); part1 = in1 && (e1 & 1);
    if (in0) ++i0;
    if (in1) ++i1;
    return true;
  }
};

// CTA -> (sequence, K/V head, two sub-tiles); longest query tiles first.
__device__ __forceinline__ void cta_work(const Params& p, int cta, int& b, int& g, SubTile (&st)[2]) {
  const int G = p.G, nrt = p.n_row_tiles;
  int h[2], rt[2];
  bool present[2];
  if (G >= 2) {
    const int PP = (G + 1) / 2;
    const int per = p.n_seq * p.Hkv * PP;
    const int r_t = nrt - 1 - cta / per;
    int r = cta % per;
    const int pp = r % PP;
    r /= PP;
    g = r % p.Hkv;
    b = r / p.Hkv;
    for (int t = 0; t < 2; ++t) {
      int hh = 2 * pp + t;
      present[t] = hh < G;
      h[t] = g * G + (present[t] ? hh : 0);
      rt[t] = r_t;
    }
  } else {
    const int NR2 = (nrt + 1) / 2;
    const int per = p.n_seq * p.Hq;
    const int rp = NR2 - 1 - cta / per;
    const int r = cta % per;
    const int hq = r % p.Hq;
    b = r / p.Hq;
    g = hq;
    for (int t = 0; t < 2; ++t) {
      rt[t] = 2 * rp + t;
      present[t] = rt[t] < nrt;
      h[t] = hq;
    }
  }
  for (int t = 0; t < 2; ++t) {
    st[t].h = h[t];
    st[t].rt = rt[t];
    st[t].valid = false;
    st[t].count = 0;
    st[t].tiles = nullptr;
    if (present[t]) {
      int64_t item = ((int64_t)b * p.Hq + h[t]) * p.n_row_tiles + rt[t];
      int c = p.item_count[item];
      st[t].valid = c >= 0;
      st[t].count = c > 0 ? c : 0;
      st[t].tiles = p.item_tiles + item * p.n_kt;
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
// a + b rounded toward minus infinity
__device__ __forceinline__ float2 add2_rm(float2 a, float2 b) {
  uint64_t d;
  asm("add.rm.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// 2^v for a pair, on the FMA and integer pipes instead of the special-function
// unit, whose 16 results per clock and SM would otherwise bound the softmax.
// v = n + f with n = floor(v), f in [0, 1); 2^f ~ 1 + f (c1 + f (c2 + f c3)),
// a minimax cubic for the relative error (at most 8.6e-5, below the 2^-9
// rounding of the bf16 P it feeds), fitted by exp2_fit.py in this package;
// n is added to the exponent field.  v is clamped at -127, where the result is
// exactly 0.  Only used where v <= 8 is known (FULL tiles, lazy rescale bound).
constexpr float kExp2C1 = 6.951167865e-01f;
constexpr float kExp2C2 = 2.276449909e-01f;
constexpr float kExp2C3 = 7.706704220e-02f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: ulp 1, so v + it rounds v to an integer
__device__ __forceinline__ float2 exp2_poly2(float2 v) {
  v.x = fmaxf(v.x, -127.f);
  v.y = fmaxf(v.y, -127.f);
  const float2 magic = make_float2(kRoundMagic, kRoundMagic);
  const float2 t = add2_rm(v, magic);        // floor(v) + magic, exact
  const float2 f = sub2(v, sub2(t, magic));  // v - floor(v), exact
  float2 q = fma2(make_float2(kExp2C3, kExp2C3), f, make_float2(kExp2C2, kExp2C2));
  q = fma2(q, f, make_float2(kExp2C1, kExp2C1));
  q = fma2(q, f, make_float2(1.f, 1.f));
  // the low mantissa bits of t hold floor(v); shifted by 23 they add it to the
  // exponent of q (the magic's own bits shift out)
  return make_float2(__int_as_float(__float_as_int(q.x) + (__float_as_int(t.x) << 23)),
                     __int_as_float(__float_as_int(q.y) + (__float_as_int(t.y) << 23)));
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 128 values held as 64 pairs: a tree of three-input maxima over
// four independent accumulators.
__device__ __forceinline__ float row_max128(const float2 (&x)[64]) {
  float m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) m[k] = fmaxf(x[k].x, x[k].y);
#pragma unroll
  for (int i = 4; i < 64; ++i) m[i & 3] = max3f(m[i & 3], x[i].x, x[i].y);
  return max3f(fmaxf(m[0], m[1]), m[2], m[3]);
}

__device__ __forceinline__ void fail(const Params& p, volatile int* abort_flag, uint32_t where) {
  if (!*abort_flag) {
    *abort_flag = 1;
    record_error(p, FA_ERR_DEVICE_TIMEOUT, where);
  }
}

// Output pointers of query row i (within its sequence) for q-head h.
__device__ __forceinline__ void row_out(const Params& p, int b, int h, int i, uint16_t*& optr, float*& lptr) {
  int64_t qrow = p.cu_q ? (int64_t)p.cu_q[b] + i : (int64_t)i;
  int64_t bo = p.cu_q ? 0 : (int64_t)b;
  optr = p.o + bo * p.o_sb + qrow * p.o_ss + (int64_t)h * p.o_sh;
  lptr = p.lse + bo * p.lse_sb + (int64_t)h * p.lse_sh + qrow * p.lse_ss;
}

template <int D>
__device__ __forceinline__ void write_empty_row(const Params& p, int b, int h, int i) {
  uint16_t* optr;
  float* lptr;
  row_out(p, b, h, i, optr, lptr);
#pragma unroll
  for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(optr + c) = make_uint4(0, 0, 0, 0);
  *lptr = -INFINITY;
}

// Per-row key range allowed by the pair rules (causal bottom-right, window,
// key bound), inclusive; empty (lo > hi) for rows past the sequence end.
__device__ __forceinline__ void row_key_range(const Params& p, int i, int q_len, int kv_len, int off, int& lo,
                                              int& hi) {
  lo = 0;
  hi = kv_len - 1;
  if (p.causal) hi = min(hi, i + off);
  if (p.wl >= 0) lo = max(lo, i + off - p.wl);
  if (p.wr >= 0) hi = min(hi, i + off + p.wr);
  if (i >= q_len) { lo = 1; hi = 0; }
}

// MK: additive term kind (FA_MASK_NONE / DENSE / TOPK); SC: logit soft-cap on.
template <int D, int MK, bool SC>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const Params p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using C = PCfg<D>;
  constexpr int NS = C::NS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int b, g;
  SubTile st[2];
  cta_work(p, blockIdx.x, b, g, st);
  if (!st[0].valid && !st[1].valid) return;
  const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
  const int off = kv_len - q_len;

  // Nothing scheduled for either sub-tile: only zero rows to write.
  if (st[0].count == 0 && st[1].count == 0) {
    if (warp >= 4) {
      const int t = (warp - 4) >> 2;
      const int i = st[t].rt * 128 + 32 * (warp & 3) + lane;
      if (st[t].valid && i < q_len) write_empty_row<D>(p, b, st[t].h, i);
    }
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NS;
  uint64_t* k_empty = v_full + NS;
  uint64_t* v_empty = k_empty + NS;
  uint64_t* s_full = v_empty + NS;    // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* o_final = p_full + 2;     // [2]
  uint64_t* mma_done = o_final + 2;   // [2]
  uint64_t* tok = mma_done + 2;       // [2] issue-order token between the MMA issuers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tok + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (tid == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(k_empty + s, 2);  // one arrival per MMA issuer
      tc::mbar_init(v_empty + s, 2);
    }
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(s_full + t, 1);
      tc::mbar_init(p_full + t, 128);
      tc::mbar_init(o_final + t, 1);
      tc::mbar_init(mma_done + t, 1);
      tc::mbar_init(tok + t, 1);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (warp == 0 || warp == 2) {
      // ---------------------------------------------------------- producers
      // warp 0: Q once, then K tiles; warp 2: V tiles.  Each ring has its own
      // release barrier: a K stage frees when the QKs that read it are done,
      // a V stage when its PVs are done, a step later.
      if (lane == 0) {
        const bool is_k = (warp == 0);
        const int kv_row0 = p.cu_k ? p.cu_k[b] : 0;
        const int kv_b = p.cu_k ? 0 : b;
        const CUtensorMap* map = is_k ? &tmk : &tmv;
        uint64_t* full = is_k ? k_full : v_full;
        uint64_t* empty = is_k ? k_empty : v_empty;
        unsigned char* ring = smem + (is_k ? C::kKOff : C::kVOff);
        tc::tma_prefetch_desc(map);
        if (is_k) {
          const int q_row0 = p.cu_q ? p.cu_q[b] : 0;
          const int q_b = p.cu_q ? 0 : b;
          tc::tma_prefetch_desc(&tmq);
          uint32_t qbytes = 0;
          for (int t = 0; t < 2; ++t)
            if (st[t].count > 0) qbytes += C::kTileBytes;
          tc::mbar_arrive_expect_tx(q_full, qbytes);
          for (int t = 0; t < 2; ++t) {
            if (st[t].count == 0) continue;
            unsigned char* dst = smem + C::kQOff + t * C::kTileBytes;
            for (int c = 0; c < D / 64; ++c)
              tc::tma_load_4d(dst + c * 16384, &tmq, q_full, c * 64, st[t].h, q_row0 + st[t].rt * 128, q_b);
          }
        }
        Merge m;
        m.init(st);
        int kt, j = 0;
        bool in0, in1, pa0, pa1;
        while (m.next(kt, in0, in1, pa0, pa1)) {
          const int s = j % NS;
          if (j >= NS && !tc::mbar_wait(empty + s, ((j / NS) - 1) & 1, abort_flag)) {
            fail(p, abort_flag, is_k ? 1 : 7);
            break;
          }
          tc::mbar_arrive_expect_tx(full + s, C::kTileBytes);
          for (int c = 0; c < D / 64; ++c)
            tc::tma_load_4d(ring + s * C::kTileBytes + c * 16384, map, full + s, c * 64, g, kv_row0 + kt * 128,
                            kv_b);
          ++j;
        }
        if (*abort_flag) {
          // let the copies already issued land before the CTA can exit
          const int first = j > NS ? j - NS : 0;
          for (int jj = first; jj < j; ++jj) tc::mbar_wait_drain(full + jj % NS, (jj / NS) & 1, 100000000ull);
          if (is_k) tc::mbar_wait_drain(q_full, 0, 100000000ull);
        }
      }
    } else if (warp == 1 || warp == 3) {
      // ---------------------------------------------------------- MMA issuers
      // The MMA queue is shallow: an issuing thread stalls on tcgen05.mma almost
      // at once, so whatever a lone issuer does between its MMA groups (waits,
      // list walk, commits) is tensor idle time.  Two issuers, one per sub-tile
      // (warp 1: sub-tile 0, warp 3: sub-tile 1), hand a token back and forth so
      // that the groups still go out in the order PV_0 QK_0 | PV_1 QK_1 | PV_0 ...
      // (the ping-pong of the two softmax warpgroups) while each one's
      // bookkeeping overlaps the other's MMAs.  Both walk the merged tile list,
      // which the K/V rings follow; a stage is released once both are done with
      // it (arrival count 2).
      auto issue = [&](auto T) {
        constexpr int t = decltype(T)::value;
        constexpr uint32_t idS = tc::idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t idO = tc::idesc_bf16_f32(128, D, false, true);
        const uint32_t sQ = tc::smem_u32(smem + C::kQOff + t * C::kTileBytes);
        const uint32_t sK = tc::smem_u32(smem + C::kKOff);
        const uint32_t sV = tc::smem_u32(smem + C::kVOff);
        const uint32_t tS = tbase + t * 128, tO = tbase + C::kOCol + t * D;
        bool ok = tc::mbar_wait(q_full, 0, abort_flag);
        if (!ok) fail(p, abort_flag, 2);
        tc::fence_after_sync();
        int prev = -1;        // merged index of this sub-tile's last QK; its PV is pending
        bool o_acc = false;   // O already holds a partial sum
        uint32_t pph = 0, tph = 0;
        auto do_pv = [&]() -> bool {
          const int ps = prev % NS;
          if (!tc::mbar_wait(p_full + t, pph, abort_flag)) return false;
          pph ^= 1;
          tc::fence_after_sync();
          const uint32_t vbase = sV + ps * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_ts(tO, tS + ks * 8, tc::sdesc_sw128(vbase + ks * 2048, 16384, 1024), idO,
                       (o_acc || ks > 0) ? 1u : 0u);
          o_acc = true;
          tc::mma_commit(v_empty + ps);
          return true;
        };
        Merge m;
        m.init(st);
        int kt, j = 0;
        bool in[2], pa[2];
        while (ok && m.next(kt, in[0], in[1], pa[0], pa[1])) {
          const int s = j % NS;
          const bool mine = t ? in[1] : in[0];
          // the stages of this entry (and, for a PV, of the previous own one)
          if (!tc::mbar_wait(k_full + s, (j / NS) & 1, abort_flag)) { ok = false; break; }
          if (prev >= 0 && mine && !tc::mbar_wait(v_full + prev % NS, (prev / NS) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (!mine && !tc::mbar_wait(v_full + s, (j / NS) & 1, abort_flag)) { ok = false; break; }
          // the partner's group for the previous entry (sub-tile 1: for this one)
          if (t == 1 || j > 0) {
            if (!tc::mbar_wait(tok + t, tph, abort_flag)) { ok = false; break; }
            tph ^= 1;
          }
          if (mine) {
            if (prev >= 0 && !do_pv()) { ok = false; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
              tc::mma_ss(tS, tc::sdesc_sw128(sQ + o, 16, 1024),
                         tc::sdesc_sw128(sK + s * C::kTileBytes + o, 16, 1024), idS, ks > 0 ? 1u : 0u);
            }
            tc::mma_commit(s_full + t);
            prev = j;
          }
          tc::mbar_arrive(tok + (1 - t));  // this entry's group is issued
          tc::mma_commit(k_empty + s);
          if (!mine) tc::mma_commit(v_empty + s);
          ++j;
        }
        if (ok && prev >= 0) {
          ok = tc::mbar_wait(v_full + prev % NS, (prev / NS) & 1, abort_flag) && do_pv();
          if (ok) tc::mma_commit(o_final + t);
        }
        if (!ok) fail(p, abort_flag, 3);
        // drain: nothing issued may still run when TMEM is released
        tc::mma_commit(mma_done + t);
        tc::mbar_wait_drain(mma_done + t, 0, 200000000ull);
      };
      if (lane == 0) {
        if (warp == 1) issue(std::integral_constant<int, 0>{});
        else issue(std::integral_constant<int, 1>{});
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int wtid = tid - 128 - 128 * t;  // 0..127 within the warpgroup
    const int wq = warp & 3;               // TMEM lane quarter this warp may access
    const int row = 32 * wq + lane;
    const SubTile me = st[t];
    const int i = me.rt * 128 + row;
    const int h = me.h;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * wq) << 16);
    const uint32_t scol = lane_base + t * 128;
    int jlo_r, jhi_r;
    row_key_range(p, i, q_len, kv_len, off, jlo_r, jhi_r);
    // top-k: per key tile, the keys' expiry rows and bias, staged in smem
    int2* kbuf = reinterpret_cast<int2*>(smem + C::kBarOff + 256) + t * 256;
    if (me.valid && me.count == 0) {
      if (i < q_len) write_empty_row<D>(p, b, h, i);
    } else if (me.valid) {
      float m_ref = -INFINITY, l = 0.f;
      uint32_t sph = 0;
      bool first = true, ok = true;
      int par = 0;
      Merge m;
      m.init(st);
      int kt;
      bool in[2], pa[2];
      while (m.next(kt, in[0], in[1], pa[0], pa[1])) {
        const bool mine = t ? in[1] : in[0];
        const bool part = t ? pa[1] : pa[0];
        if (!mine) continue;
        const int j0 = kt * kKeysPerTile;
        if (MK == FA_MASK_TOPK) {
          const int jj = j0 + wtid;
          int2 v = make_int2(kRowNever, 0);
          if (jj < kv_len) {
            const int64_t bh = (int64_t)b * p.Hq + h;
            v.x = __ldg(p.topk_e + bh * p.Sk + jj);
            v.y = __float_as_int(
                __ldg(p.z + (int64_t)b * p.z_sb + (int64_t)h * p.z_sh + (int64_t)jj * p.z_sk) * kLog2e);
          }
          kbuf[par * 128 + wtid] = v;
          asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
        }
        if (!tc::mbar_wait(s_full + t, sph, abort_flag)) { ok = false; break; }
        sph ^= 1;
        tc::fence_after_sync();
        float2 x[64];
        {
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tc::tmem_ld32(scol + c * 32, r[c]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              x[c * 16 + e] = make_float2(__uint_as_float(r[c][2 * e]), __uint_as_float(r[c][2 * e + 1]));
        }
        // logits in log2 units; a FULL tile without soft-cap keeps raw scores
        // and folds the scale into the exponent below
        const bool plain = !SC && !part;
        float mx;
        if (plain) {
          mx = row_max128(x) * p.scale_log2;
        } else {
          const int clo = jlo_r - j0, chi = jhi_r - j0;
          const bool all_in = !part;
          const float* mrow = nullptr;
          if (MK == FA_MASK_DENSE && i < q_len)
            mrow = p.mask + (int64_t)(p.m_nb > 1 ? b : 0) * p.m_sb + (int64_t)(p.m_nh > 1 ? h : 0) * p.m_sh +
                   (int64_t)i * p.m_sq + (int64_t)j0 * p.m_sk;
#pragma unroll
          for (int e = 0; e < 128; ++e) {
            float v = (e & 1) ? x[e >> 1].y : x[e >> 1].x;
            if (SC) {
              v = p.softcap * tanhf(v * p.scale / p.softcap) * kLog2e;
            } else {
              v = v * p.scale_log2;
            }
            bool keep = all_in || (e >= clo && e <= chi);
            if (MK == FA_MASK_DENSE && !all_in) {
              if (keep) v += __ldg(mrow + (int64_t)e * p.m_sk) * kLog2e;
            }
            if (MK == FA_MASK_TOPK) {
              const int2 kv = kbuf[par * 128 + e];
              keep = keep && (i < kv.x);
              v += __int_as_float(kv.y);
            }
            v = keep ? v : -INFINITY;
            if (e & 1) x[e >> 1].y = v; else x[e >> 1].x = v;
          }
          mx = row_max128(x);
        }
        // raise the exponent reference only when the row max outgrew it by 2^8
        const bool upd = mx > m_ref + kRescaleLog2;
        const float alpha = upd ? fast_exp2(m_ref - mx) : 1.f;
        const bool need_o = upd && !first && m_ref != -INFINITY;
        if (__any_sync(0xffffffffu, need_o)) {
          const float f = need_o ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            const uint32_t a = lane_base + C::kOCol + t * D + c * 32;
            tc::tmem_ld32(a, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
            tc::tmem_st32(a, r);
          }
          tc::tmem_wait_st();
        }
        if (upd) {
          l *= alpha;
          m_ref = mx;
        }
        const float eref = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 ner = make_float2(-eref, -eref);
        float2 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
        // P = exp2(x - ref): one packed FMA (FULL: scale folded in) or add per pair
        if (plain) {
          const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = fma2(x[c * 16 + e], sl2, ner);
              // some exponentials on the FMA pipes, interleaved with the SFU ones
              // (a warp issues in order: the ALU work fills the SFU's gaps)
              const float2 pe = false ? exp2_poly2(v) : make_float2(fast_exp2(v.x), fast_exp2(v.y));
              acc[e & 3] = add2(acc[e & 3], pe);
              pk[e] = pack2(pe.x, pe.y);
            }
            tc::tmem_st16(scol + c * 16, pk);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = add2(x[c * 16 + e], ner);
              const float2 pe = make_float2(fast_exp2(v.x), fast_exp2(v.y));
              acc[e & 3] = add2(acc[e & 3], pe);
              pk[e] = pack2(pe.x, pe.y);
            }
            tc::tmem_st16(scol + c * 16, pk);
          }
        }
        acc[0] = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
        l += acc[0].x + acc[0].y;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(p_full + t);
        first = false;
        par ^= 1;
      }
      if (ok) ok = tc::mbar_wait(o_final + t, 0, abort_flag);
      if (!ok) {
        fail(p, abort_flag, 4 + t);
      } else {
        tc::fence_after_sync();
        const bool empty = !(l > 0.f);
        const float inv = empty ? 0.f : 1.f / l;
        uint16_t* optr;
        float* lptr;
        row_out(p, b, h, i < q_len ? i : 0, optr, lptr);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(lane_base + C::kOCol + t * D + c * 32, r);
          tc::tmem_wait_ld();
          if (i < q_len) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack2(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
              w.y = pack2(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
              w.z = pack2(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
              w.w = pack2(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
              *reinterpret_cast<uint4*>(optr + c * 32 + 8 * v4) = w;
            }
          }
        }
        if (i < q_len) *lptr = empty ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tbase, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 4-D map {d, heads, rows, batch} over a bshd (or packed thd) bf16 tensor,
// box {64, 1, 128, 1}, 128-byte swizzle; rows beyond the tensor read as 0.
bool encode_bshd(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int batch, int64_t s_h,
                 int64_t s_row, int64_t s_b) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)s_h * 2, (cuuint64_t)s_row * 2, (cuuint64_t)s_b * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int MK, bool SC>
cudaError_t launch_prefill_v(const Params& p, cudaStream_t st, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, int64_t grid, cudaEvent_t ev_begin) {
  auto kern = prefill_kernel<D, MK, SC>;
  // setmaxnreg.inc would wait forever if the block were launched with fewer
  // registers than the split assumes: launch only when the build matches.
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaError_t e = ensure_smem_attr<prefill_kernel<D, MK, SC>>(PCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  if (ev_begin && (e = cudaEventRecord(ev_begin, st)) != cudaSuccess) return e;
  kern<<<(unsigned)grid, kPrefillThreads, PCfg<D>::kSmem, st>>>(p, mq, mk, mv);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_d(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  CUtensorMap mq, mk, mv;
  const bool vq = p.cu_q != nullptr, vk = p.cu_k != nullptr;
  // extents of 1 get a harmless stride (the stride of the next-inner dimension)
  const int64_t q_rows = vq ? p.tot_q : p.Sq, k_rows = vk ? p.tot_k : p.Sk;
  const int qb = vq ? 1 : p.n_seq, kb = vk ? 1 : p.n_seq;
  const int64_t q_sb = (qb == 1 || p.q_sb == 0) ? p.q_ss : p.q_sb;
  const int64_t k_sb = (kb == 1 || p.k_sb == 0) ? p.k_ss : p.k_sb;
  const int64_t v_sb = (kb == 1 || p.v_sb == 0) ? p.v_ss : p.v_sb;
  if (!encode_bshd(&mq, p.q, D, p.Hq, q_rows, qb, p.q_sh, p.q_ss, q_sb) ||
      !encode_bshd(&mk, p.k, D, p.Hkv, k_rows, kb, p.k_sh, p.k_ss, k_sb) ||
      !encode_bshd(&mv, p.v, D, p.Hkv, k_rows, kb, p.v_sh, p.v_ss, v_sb))
    return cudaErrorInvalidValue;
  int64_t grid;
  if (p.G >= 2)
    grid = (int64_t)p.n_row_tiles * p.n_seq * p.Hkv * ((p.G + 1) / 2);
  else
    grid = (int64_t)((p.n_row_tiles + 1) / 2) * p.n_seq * p.Hq;
  if (grid <= 0) return ev_begin ? cudaEventRecord(ev_begin, st) : cudaSuccess;
  const bool sc = p.softcap > 0.f;
  switch (p.mask_kind) {
    case FA_MASK_DENSE:
      return sc ? launch_prefill_v<D, FA_MASK_DENSE, true>(p, st, mq, mk, mv, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_DENSE, false>(p, st, mq, mk, mv, grid, ev_begin);
    case FA_MASK_TOPK:
      return sc ? launch_prefill_v<D, FA_MASK_TOPK, true>(p, st, mq, mk, mv, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_TOPK, false>(p, st, mq, mk, mv, grid, ev_begin);
    default:
      return sc ? launch_prefill_v<D, FA_MASK_NONE, true>(p, st, mq, mk, mv, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_NONE, false>(p, st, mq, mk, mv, grid, ev_begin);
  }
}

}  // namespace

cudaError_t launch_prefill(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  if (p.n_items <= 0) return ev_begin ? cudaEventRecord(ev_begin, st) : cudaSuccess;
  if (p.d == 64) return launch_prefill_d<64>(p, st, ev_begin);
  return launch_prefill_d<128>(p, st, ev_begin);
}

}  // namespace mfa
