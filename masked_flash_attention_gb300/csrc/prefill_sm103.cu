// prefill_sm103.cu -- masked flash-attention forward for many query rows on
// the 5th-generation tensor cores of sm_103a (tcgen05 + TMEM + TMA).
//
// The method is the tiled, online-softmax attention of the ExecuTorch pull
// request 10466 "Summary": q@k is cut into chunks along both the query and the
// key dimension, the softmax is accumulated progressively and rescaled at the
// end; an all -inf chunk must not poison the running values.  Chunks whose
// every pair is masked are not computed at all: with a dense or top-k mask the
// scheduler (sched.cu, topk.cu) left them out of each item's key-tile list;
// without one the kernel derives each unit's tiles from its geometry.
//
// Persistent kernel: one CTA per SM (two at d = 64) walks the work units (sequence, q-head,
// 128-row query tile) longest first, in rounds of one unit per CTA with every
// other round in reverse CTA order (serpentine), so the pipelines run on from
// one unit into the next (Q of the next unit is fetched while the current one
// runs, or at d = 128 once its QKs are done; its first QK overlaps the current
// epilogue).
// When the last round would hold at most half the grid (a causal launch over
// past keys: 512 units of almost equal length on 152 CTAs leave 56 for the
// fourth round), each of its units is cut in two over its key tiles and run
// by two CTAs; the two pieces' normalised rows are merged by their
// log-sum-exp, the same rescaling the chunked softmax uses across chunks,
// by whichever piece finishes second.
// Grouped-query heads read their K/V head directly (InfiniTrain pull request
// 193 "Transformer 接入": no expansion); neighbouring units are the q-heads of
// one group, so their K/V tiles are served from L2.
//
// Warp roles (12 warps; 16 in the top-k variants; 8 at d = 64 otherwise):
//   warp 0      TMA producer: K tiles through an NSK-stage ring
//   warp 1      QK issuer (one thread), Q prefetch, TMEM owner
//   warp 2      TMA producer: V tiles through an NSV-stage ring
//   warp 3      PV issuer (one thread)
//   warps 4..7  softmax warpgroup 0: the even key tiles of a unit's sequence
//   warps 8..11 softmax warpgroup 1: the odd ones
//   warps 12..15 (top-k) more K and V gather issuers
// TMEM (512 columns): S in two buffers [0,128) [128,256) (fp32), P in two
// buffers [256,320) [320,384) (input type, two per column), O in [384, 384 + D).
// With S and P double-buffered QK(j+1) runs while the softmax of tile j does,
// and PV(j) while the softmax of tile j+1 does; the tensor cores wait on the
// softmax only when it is slower than QK + PV.  The MMA queue is shallow (an
// issuing thread stalls on tcgen05.mma almost at once), so QK and PV come from
// two threads: each one's waits overlap the other's MMAs.
// The two softmax warpgroups take alternate key tiles of the same 128 rows;
// each thread owns one whole 128-key row of its tile (32x32b TMEM loads).  The
// exponent reference of a row is handed from tile to tile through shared
// memory, and the two warpgroups' row sums are added at the end.  The
// reference is only raised when the row max exceeds it by more than 2^8 (in
// log2 units), so O in TMEM is rarely rescaled.  A fully masked row keeps reference -inf,
// exponentiates against 0, and ends with l = 0: O = 0, LSE = -inf.
// At d = 64 (no top-k) the tiles are short and a unit's fixed costs weigh
// most, so a CTA has a single softmax warpgroup (warps 4..7, every tile of
// its units) and 256 TMEM columns (S [0,128), P [128,192), O [192,256)), and
// two CTAs share each SM: one CTA's unit epilogue overlaps the other's tiles.
//
// Every mbarrier wait is bounded (1 s); on a time-out the kernel records
// FA_ERR_DEVICE_TIMEOUT in the workspace error word, every role stops, in-flight
// MMAs are drained and TMEM is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>

#include "fa_device.cuh"
#include "host_util.h"
#include "tc_sm103.cuh"

namespace mfa {

namespace {

constexpr int kPrefillThreads = 384;
// The top-k variants gather their key rows with TMA tile::gather4, which one
// warp issues at only about one copy per 65-90 cycles; they launch a fourth
// warpgroup (warps 12..15) whose warps share the K and V gathers with the two
// producer warps, three warps per operand.
constexpr int kGatherThreads = 512;
// Register split (setmaxnreg): the kernel is built to launch with exactly
// kLaunchRegs per thread (kGatherLaunchRegs for the top-k variants);
// warpgroup 0 (producers, issuers) and the gather warpgroup give registers
// back and the two softmax warpgroups take them, so that a 128-key row of S
// fits in registers.
constexpr int kLaunchRegs = 168;
constexpr int kGatherLaunchRegs = 128;
constexpr int kProducerRegs = 72;
constexpr int kGatherProducerRegs = 40;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kProducerRegs + 256 * kSoftmaxRegs <= kPrefillThreads * kLaunchRegs,
              "the register split must fit the block's launch allocation");
static_assert(256 * kGatherProducerRegs + 256 * kSoftmaxRegs <= kGatherThreads * kGatherLaunchRegs,
              "the register split must fit the block's launch allocation");
// At d = 64 (no top-k) a CTA has one softmax warpgroup (8 warps) and two
// CTAs share each SM: half the TMEM and shared memory each, and the same
// 40 / 216 register split as the gather variants.
constexpr int kPairThreads = 256;
__host__ __device__ constexpr int prefill_threads(int d, int mk) {
  return mk == FA_MASK_TOPK ? kGatherThreads : (d == 64 ? kPairThreads : kPrefillThreads);
}
__host__ __device__ constexpr int prefill_launch_regs(int d, int mk) {
  return (mk == FA_MASK_TOPK || d == 64) ? kGatherLaunchRegs : kLaunchRegs;
}
__host__ __device__ constexpr int prefill_ctas_per_sm(int d, int mk) { return (d == 64 && mk != FA_MASK_TOPK) ? 2 : 1; }
static_assert(128 * kGatherProducerRegs + 128 * kSoftmaxRegs <= kPairThreads * kGatherLaunchRegs,
              "the register split must fit the block's launch allocation");
static_assert(2 * kPairThreads * kGatherLaunchRegs <= 65536, "two CTAs per SM must fit the register file");
constexpr float kRescaleLog2 = 8.0f;

template <int D, bool GTH = false>
struct PCfg {
  // Softmax warpgroups per CTA.  Two take alternate key tiles of one unit
  // (S and P double-buffered in TMEM).  At d = 64 without top-k a CTA has
  // one, which takes every tile of its units, and two CTAs run on each SM:
  // a unit's epilogue in one CTA (waiting for its last PV, normalising,
  // storing) then overlaps the other CTA's tiles instead of stalling the
  // SM's tensor pipe, as a shared O buffer would.
  static constexpr int NW = (D == 64 && !GTH) ? 1 : 2;
  // TMEM: S buffers (128 fp32 columns each), P buffers (128 keys of the
  // input type, two per column) and O; 512 columns, 256 with NW == 1.
  static constexpr uint32_t kCols = NW == 2 ? 512 : 256;
  static constexpr uint32_t kSCol = 0;              // S buffer b: kSCol + 128 * b
  static constexpr uint32_t kPCol = 128 * NW;       // P buffer b: kPCol + 64 * b
  static constexpr uint32_t kOCol = kPCol + 64 * NW;
  // Ring stages and Q buffers.  At d = 128 a third K stage (so that a K
  // tile's copy has a tile period more to land before its QK) is paid for
  // with the second Q buffer: the next unit's Q is then fetched once the
  // current unit's QKs are done, which the epilogue hides (the causal-prefill
  // workload 124.3 -> 114.7 us, the Llama-3 layer 408 -> 376 us).  The
  // gathered top-k tiles keep two Q buffers and two K stages (with three K
  // stages and one Q buffer they measured 371 us against 351 us).  With two
  // CTAs per SM each has two of everything.
  static constexpr int NQ = (D == 128 && !GTH) ? 1 : 2;                          // Q buffers
  static constexpr int NSK = (D == 128) ? (GTH ? 2 : 3) : (NW == 1 ? 2 : 4);     // K ring stages
  static constexpr int NSV = (D == 128 || NW == 1) ? 2 : 4;                      // V ring stages
  static constexpr int kTileBytes = 128 * D * 2;    // one 128-row tile of 2-byte elements
  static constexpr int kQOff = 0;                   // NQ Q buffers
  static constexpr int kKOff = NQ * kTileBytes;
  static constexpr int kVOff = kKOff + NSK * kTileBytes;
  static constexpr int kAuxOff = kVOff + NSV * kTileBytes;
  // aux: barriers and flags (512 B), row references [2][128] floats, row
  // sums [2][128] floats, top-k staging [2 warpgroups][2 buffers]
  static constexpr int kRedOff = kAuxOff + 512;
  static constexpr int kSumOff = kRedOff + 2 * 128 * 4;
  static constexpr int kTopkOff = kSumOff + 2 * 128 * 4;
  // top-k staging, per warpgroup and buffer: first keeping row, number of
  // keeping rows (int) and bias (fp32) of each of the tile's 128 columns
  static constexpr int kTopkBuf = 3 * 128 * 4;
  // output staging: per softmax warp 32 rows x 32 output columns
  static constexpr int kStageOff = (kTopkOff + (GTH ? 2 * 2 * kTopkBuf : 0) + 1023) / 1024 * 1024;  // swizzle-aligned
  static constexpr int kSmem = kStageOff + 4 * NW * 2048 + 1024;  // + alignment slack
  static_assert(kSmem <= (NW == 2 ? 227 * 1024 : 113 * 1024), "shared memory budget");
  static_assert(kStageOff % 1024 == 0, "TMA store source alignment");
  static_assert(kOCol + D <= kCols, "TMEM budget");
};

// One work unit: 128 query rows of one q-head of one sequence.  Its key tiles
// come from the scheduler kernel's list, or -- when the pair rules alone decide
// them (no dense or top-k mask: INL, the host's p.sched_inline) -- from the
// unit's geometry: tiles kt0 .. kt0 + count - 1, those with relative index in
// [fl, fh] FULL and the others PARTIAL, exactly what the scheduler kernel
// would have listed.
// A slot of a split last round (INL only, Params::tail_units) holds one of
// the two pieces of a unit: a unit over half of its key tiles.
struct Unit {
  bool present;  // the tile holds rows of the sequence
  bool valid;    // the sequence's lengths passed the checks
  int b, h, rt, count;
  int kt0, fl, fh;       // INL
  const int32_t* tiles;  // scheduler list (not INL)
};

// Floor of a / 128 for any sign of a.
__device__ __forceinline__ int floor_div128(int a) { return a >= 0 ? a / 128 : -((127 - a) / 128); }

// Unit u, longest query tiles first (row tile descending), q-heads fastest.
template <bool INL, bool GTH = false>
__device__ __forceinline__ Unit unit_of(const Params& p, int u) {
  Unit w;
  const int q = fast_div(u, p.div_units);
  w.rt = p.n_row_tiles - 1 - q;
  const int r = u - q * (p.n_seq * p.Hq);
  w.b = fast_div(r, p.div_hq);
  w.h = r - w.b * p.Hq;
  const int q_len = seq_qlen(p, w.b);
  w.present = w.rt * 128 < q_len;
  if constexpr (INL) {
    const int kv_len = seq_klen(p, w.b);
    w.valid = !seq_lengths_bad(p, w.b, q_len, kv_len);
    w.count = 0;
    w.kt0 = 0;
    w.fl = 1;
    w.fh = 0;
    if (w.valid && w.present && kv_len > 0) {
      const int i0 = w.rt * 128, i1 = min(i0 + 127, q_len - 1), off = kv_len - q_len;
      int jlo = 0, jhi = kv_len - 1;
      const bool no_skip = (p.debug_flags & FA_DEBUG_NO_SKIP) != 0;
      if (!no_skip) key_range(p, i0, i1, off, kv_len, jlo, jhi);
      if (jlo <= jhi) {
        w.kt0 = jlo / kKeysPerTile;
        w.count = jhi / kKeysPerTile - w.kt0 + 1;
        if (!no_skip) {
          // tile_all_allowed as a range of tiles: the last key of the tile at
          // most hi, its first key at least lo
          int hi = kv_len - 1, lo = INT_MIN / 2;
          if (p.causal) hi = min(hi, i0 + off);
          if (p.wr >= 0) hi = min(hi, i0 + off + p.wr);
          if (p.wl >= 0) lo = i1 + off - p.wl;
          const int kt_hi = floor_div128(hi - (kKeysPerTile - 1));
          const int kt_lo = lo <= 0 ? 0 : -floor_div128(-lo);
          w.fl = max(kt_lo, w.kt0) - w.kt0;
          w.fh = kt_hi - w.kt0;
        }
      }
    }
  } else {
    const int64_t item = ((int64_t)w.b * p.Hq + w.h) * p.n_row_tiles + w.rt;
    const int c = w.present ? __ldg(p.item_count + item) : -1;
    w.valid = c >= 0;
    w.count = c > 0 ? c : 0;
    w.tiles = p.item_tiles + item * p.n_kt;
    if constexpr (GTH) w.fl = w.present ? __ldg(p.topk_full + item) : 0;  // leading FULL gathered tiles
  }
  return w;
}

// The piece slot `slot` holds: 0 for a whole unit; with a tail split, slot
// t0 + k of the last round (t0 = tail_round * grid) holds piece 1 + (k & 1)
// of tail unit tu = k >> 1, unit t0 + tu.
template <bool INL>
__device__ __forceinline__ int tail_piece(const Params& p, int slot, int& tu) {
  tu = 0;
  if (!INL || p.tail_units <= 0) return 0;  // the host splits d = 128 launches only
  const int t0 = p.tail_round * (int)gridDim.x;
  if (slot < t0) return 0;
  tu = (slot - t0) >> 1;
  return 1 + ((slot - t0) & 1);
}

// The unit (or piece) of slot `slot`.  The first piece of a split unit takes
// its first ceil(count / 2) key tiles, the second the rest, as a unit whose
// tiles start that many later; a unit of fewer than two tiles is not split
// (its first piece takes it whole, its second is empty).
template <bool INL, bool GTH = false>
__device__ __forceinline__ Unit unit_at(const Params& p, int slot) {
  int tu;
  const int piece = tail_piece<INL>(p, slot, tu);
  if (piece == 0) return unit_of<INL, GTH>(p, slot);
  Unit w = unit_of<INL, GTH>(p, p.tail_round * (int)gridDim.x + tu);
  if (w.present && w.valid && w.count >= 2) {
    const int h1 = (w.count + 1) >> 1;
    if (piece == 1) {
      w.count = h1;
    } else {
      w.kt0 += h1;
      w.fl -= h1;
      w.fh -= h1;
      w.count -= h1;
    }
  } else if (piece == 2) {
    w.present = false;
  }
  return w;
}

// Entry i of a unit's key-tile list: (key tile << 1) | PARTIAL.  A top-k
// unit's tiles are gathered keys (GTH): always PARTIAL, no key tile.
template <bool INL, bool GTH = false>
__device__ __forceinline__ int unit_entry(const Unit& w, int i) {
  if constexpr (GTH) return i < w.fl ? 0 : 1;
  else if constexpr (INL) return ((w.kt0 + i) << 1) | ((i < w.fl || i > w.fh) ? 1 : 0);
  else return __ldg(w.tiles + i);
}

// The gathered keys of a top-k unit: n_kt * 128 entries (x = key index |
// first keeping row << 16 | first row past the keeping ones << 24, rows
// relative to the unit's tile; y = bias in log2 units); count * 128 are set.
__device__ __forceinline__ const uint2* unit_glist(const Params& p, const Unit& w) {
  const int64_t item = ((int64_t)w.b * p.Hq + w.h) * p.n_row_tiles + w.rt;
  return p.topk_list + item * ((int64_t)p.n_kt * kKeysPerTile);
}

// Inline scheduling: the scheduler's counters (tiles scheduled FULL and
// PARTIAL, key tiles left out as EMPTY) over every unit of the launch, and
// the length checks of every sequence, by one warp.  Units of one (sequence,
// row tile) differ only in the q-head, so each pair is counted once, times Hq.
__device__ __noinline__ void inline_sched_stats(const Params& p) {
  const int lane = threadIdx.x & 31;
  unsigned long long nf = 0, np = 0, ne = 0;
  const int64_t n = (int64_t)p.n_seq * p.n_row_tiles;
  for (int64_t t = lane; t < n; t += 32) {
    const int b = (int)(t / p.n_row_tiles), rt = (int)(t % p.n_row_tiles);
    const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
    if (seq_lengths_bad(p, b, q_len, kv_len)) {
      if (rt == 0) record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)b);
      continue;
    }
    const int i0 = rt * 128;
    if (i0 >= q_len || kv_len <= 0) continue;
    const int i1 = min(i0 + 127, q_len - 1), off = kv_len - q_len;
    const int n_kt_b = (kv_len + kKeysPerTile - 1) / kKeysPerTile;
    const bool no_skip = (p.debug_flags & FA_DEBUG_NO_SKIP) != 0;
    int jlo = 0, jhi = kv_len - 1;
    if (!no_skip) key_range(p, i0, i1, off, kv_len, jlo, jhi);
    int count = 0, full = 0;
    if (jlo <= jhi) {
      const int kt0 = jlo / kKeysPerTile, kt1 = jhi / kKeysPerTile;
      count = kt1 - kt0 + 1;
      for (int kt = kt0; kt <= kt1 && !no_skip; ++kt)
        full += tile_all_allowed(p, i0, i1, kt * kKeysPerTile, kt * kKeysPerTile + kKeysPerTile - 1, off, kv_len);
    }
    nf += (unsigned long long)full * p.Hq;
    np += (unsigned long long)(count - full) * p.Hq;
    ne += (unsigned long long)(n_kt_b - count) * p.Hq;
  }
  for (int o = 16; o > 0; o >>= 1) {
    nf += __shfl_xor_sync(0xffffffffu, nf, o);
    np += __shfl_xor_sync(0xffffffffu, np, o);
    ne += __shfl_xor_sync(0xffffffffu, ne, o);
  }
  if (lane == 0) {
    p.stats[0] = nf;
    p.stats[1] = np;
    p.stats[2] = ne;
  }
}

__device__ __forceinline__ int n_units(const Params& p) { return p.n_row_tiles * p.n_seq * p.Hq; }
// Slots of the launch: one per unit, two per unit of a split last round.
__device__ __forceinline__ int n_slots(const Params& p) {
  return p.tail_units > 0 ? p.tail_round * (int)gridDim.x + 2 * p.tail_units : n_units(p);
}

// The unit this CTA takes in round r: the grid takes the units (longest
// first) in rounds of gridDim.x, every other round in reverse CTA order, so
// that the CTA taking a round's longest unit takes the next round's shortest
// (with units of falling length this balances the CTAs' loads far better
// than unit u -> CTA u mod grid).  Past the last unit in some round, a CTA is
// past it in every later round.
__device__ __forceinline__ int round_unit(int r) {
  const int c = (r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
  return r * (int)gridDim.x + c;
}

// Next round at or after r whose slot has key tiles, or -1.
template <bool INL, bool GTH = false>
__device__ __forceinline__ int next_busy(const Params& p, int r, Unit& w) {
  const int n = n_slots(p);
  for (;; ++r) {
    const int u = round_unit(r);
    if (u >= n) return -1;
    w = unit_at<INL, GTH>(p, u);
    if (w.present && w.valid && w.count > 0) return r;
  }
}

// Two fp32 values rounded to nearest-even into one packed pair of the input
// type (bf16, or fp16 when F16).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
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

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 128 values held as 64 pairs: three-input maxima over eight
// independent accumulators.
__device__ __forceinline__ float row_max128(const float2 (&x)[64]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[k].x, x[k].y);
#pragma unroll
  for (int i = 8; i < 64; ++i) m[i & 7] = max3f(m[i & 7], x[i].x, x[i].y);
  return fmaxf(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], max3f(m[5], m[6], m[7])));
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

// MK: additive term kind (FA_MASK_NONE / DENSE / TOPK); SC: logit soft-cap on;
// AL: ALiBi slopes on (only with MK == FA_MASK_NONE); F16: inputs, P and the
// output are fp16 (else bf16); DBG: the debug instantiation, which also
// writes S, P and the exponent references of one unit to Params::dump.
template <int D, int MK, bool SC, bool AL, bool F16, bool DBG = false>
__global__ void __launch_bounds__(prefill_threads(D, MK), prefill_ctas_per_sm(D, MK))
    prefill_kernel(const Params p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo, const int o_tma) {
  using C = PCfg<D, MK == FA_MASK_TOPK>;
  constexpr int NSK = C::NSK, NSV = C::NSV, NQ = C::NQ, NW = C::NW;
  constexpr uint32_t kSCol = C::kSCol, kPCol = C::kPCol, kOCol = C::kOCol;
  constexpr bool INL = (MK == FA_MASK_NONE);  // the host sets p.sched_inline exactly then
  constexpr bool GTH = (MK == FA_MASK_TOPK);   // tiles of gathered keys (2-D K/V maps)
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kAuxOff);
  uint64_t* q_full = bars;            // [2] Q buffer loaded
  uint64_t* q_empty = q_full + 2;     // [2] QKs reading a Q buffer done
  uint64_t* k_full = q_empty + 2;     // [NSK]
  uint64_t* k_empty = k_full + NSK;   // [NSK]
  uint64_t* v_full = k_empty + NSK;   // [NSV]
  uint64_t* v_empty = v_full + NSV;   // [NSV]
  uint64_t* s_full = v_empty + NSV;   // [2] S buffer written by QK
  uint64_t* s_free = s_full + 2;      // [2] S buffer read by the softmax (128 arrivals)
  uint64_t* p_full = s_free + 2;      // [2] P buffer written, O rescaled (128 arrivals)
  uint64_t* p_free = p_full + 2;      // [2] PV reading a P buffer done
  uint64_t* o_full = p_free + 2;      // [1] last PV of a unit done
  uint64_t* drained = o_full + 1;     // [2] all MMAs of an issuer done (teardown)
  uint64_t* sumx = drained + 2;       // [1] row sums of both warpgroups posted (256 arrivals)
  uint64_t* kready = sumx + 1;        // [2 warpgroups][2] top-k staging filled (128 arrivals)
  uint64_t* refb = kready + 4;        // [2 tile parity] row references posted (128 arrivals)
  uint64_t* tdone = refb + 2;         // [2 warpgroups] tail piece stored (128 arrivals)
  uint64_t* tflag = tdone + 2;        // [2 warpgroups] tail piece's merge decision posted (1 arrival)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tflag + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tsec = abort_flag + 1;  // [2 warpgroups] 1: this piece merges, 2: gave up

  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(q_full + k, 1);
      tc::mbar_init(q_empty + k, 1);
      tc::mbar_init(s_full + k, 1);
      tc::mbar_init(s_free + k, 128);
      tc::mbar_init(p_full + k, 128);
      tc::mbar_init(p_free + k, 1);
      tc::mbar_init(drained + k, 1);
      tc::mbar_init(refb + k, 128);
      tc::mbar_init(kready + k, 128);
      tc::mbar_init(kready + 2 + k, 128);
      tc::mbar_init(tdone + k, 128);
      tc::mbar_init(tflag + k, 1);
    }
    tc::mbar_init(sumx, 256);
    // gathered tiles: each of the operand's three gather warps arrives
    for (int s = 0; s < NSK; ++s) {
      tc::mbar_init(k_full + s, GTH ? 3 : 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < NSV; ++s) {
      tc::mbar_init(v_full + s, GTH ? 3 : 1);
      tc::mbar_init(v_empty + s, 1);
    }
    tc::mbar_init(o_full, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::kCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  if ((GTH || NW == 1) && (warp < 4 || warp >= 12)) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGatherProducerRegs));
  } else if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
  }
  if (GTH && (warp == 0 || warp == 2 || warp >= 12)) {
    // ------------------------------------------------------------ producers (gathered keys)
    // Three warps per operand (K: warps 0, 12, 13; V: 2, 14, 15).  A tile's
    // 128 key rows come in 32 groups of 4, each one tile::gather4 per
    // 64-column half, from the 2-D K/V view whose row b * Sk + j holds key j
    // of sequence b, every head side by side; lane l of the operand's warp
    // `part` takes row group 3 l + part.  Each warp waits for the stage to be
    // free itself and arrives on its full barrier with the bytes it sends.
    const bool is_k = warp == 0 || warp == 12 || warp == 13;
    const int part = warp < 12 ? 0 : 1 + (warp & 1);
    const int rg = 3 * lane + part;  // this lane's row group (none when >= 32)
    const uint32_t my_bytes = (uint32_t)((32 - part + 2) / 3) * (4u * D * 2u);
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    unsigned char* ring = smem + (is_k ? C::kKOff : C::kVOff);
    const int NS = is_k ? NSK : NSV;
    if (lane == 0) tc::tma_prefetch_desc(map);
    int j = 0;
    bool ok = true;
    Unit w;
    for (int r = next_busy<INL, GTH>(p, 0, w); ok && r >= 0; r = next_busy<INL, GTH>(p, r + 1, w)) {
      const int row0 = w.b * p.Sk;
      const int x0 = (w.h / p.G) * (int)(is_k ? p.k_sh : p.v_sh);
      const uint4* lst = reinterpret_cast<const uint4*>(unit_glist(p, w));
      for (int i = 0; i < w.count; ++i, ++j) {
        const int s = j % NS;
        // this lane's four keys (two entries per 16 bytes), read before the wait
        uint4 ea = make_uint4(0, 0, 0, 0), eb = ea;
        if (rg < 32) {
          ea = __ldg(lst + (i * kKeysPerTile + 4 * rg) / 2);
          eb = __ldg(lst + (i * kKeysPerTile + 4 * rg) / 2 + 1);
        }
        bool go = true;
        if (lane == 0 && j >= NS) go = tc::mbar_wait(empty + s, ((j / NS) - 1) & 1, abort_flag);
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          if (lane == 0) fail(p, abort_flag, is_k ? 1 : 7);
          ok = false;
          break;
        }
        if (lane == 0) tc::mbar_arrive_expect_tx(full + s, my_bytes);
        __syncwarp();
        if (rg < 32)
          for (int c = 0; c < D / 64; ++c)
            tc::tma_gather4_2d(ring + s * C::kTileBytes + c * 16384 + rg * 512, map, full + s, x0 + c * 64,
                               row0 + (int)(ea.x & 0xffffu), row0 + (int)(ea.z & 0xffffu),
                               row0 + (int)(eb.x & 0xffffu), row0 + (int)(eb.z & 0xffffu));
      }
    }
    if (lane == 0 && *abort_flag) {
      // let the copies already issued land before the CTA can exit
      const int first = j > NS ? j - NS : 0;
      for (int jj = first; jj < j; ++jj) tc::mbar_wait_drain(full + jj % NS, (jj / NS) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    // K (warp 0) and V (warp 2) tiles of every busy unit, in order, through
    // their rings; a stage is refilled once the MMAs that read it are done.
    if (lane == 0) {
      const bool is_k = (warp == 0);
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      unsigned char* ring = smem + (is_k ? C::kKOff : C::kVOff);
      const int NS = is_k ? NSK : NSV;
      tc::tma_prefetch_desc(map);
      // test only: the first key tile is never sent, so every wait behind it
      // runs out (FA_DEBUG_WITHHOLD)
      const bool withhold = is_k && (p.debug_flags & FA_DEBUG_WITHHOLD);
      int j = 0;
      bool ok = true;
      Unit w;
      for (int r = next_busy<INL, GTH>(p, 0, w); ok && r >= 0; r = next_busy<INL, GTH>(p, r + 1, w)) {
        const int kv_row0 = p.cu_k ? p.cu_k[w.b] : 0;
        const int kv_b = p.cu_k ? 0 : w.b;
        const int g = w.h / p.G;
        for (int i = 0; i < w.count; ++i, ++j) {
          if (withhold && j == 0) continue;
          const int kt = unit_entry<INL>(w, i) >> 1;
          const int s = j % NS;
          if (j >= NS && !tc::mbar_wait(empty + s, ((j / NS) - 1) & 1, abort_flag)) {
            fail(p, abort_flag, is_k ? 1 : 7);
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(full + s, C::kTileBytes);
          for (int c = 0; c < D / 64; ++c)
            tc::tma_load_4d(ring + s * C::kTileBytes + c * 16384, map, full + s, c * 64, g, kv_row0 + kt * 128,
                            kv_b);
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA can exit (the
        // withheld tile was never issued)
        const int first = j > NS ? j - NS : 0;
        for (int jj = first; jj < j; ++jj)
          if (!(withhold && jj == 0)) tc::mbar_wait_drain(full + jj % NS, (jj / NS) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    // S[g % NW] = Q K_g^T for the g-th tile this CTA processes, as soon as
    // the softmax has read that S buffer NW tiles back.  Also fetches Q: with two
    // buffers the next unit's Q while the current unit runs, with one the next
    // unit's Q once the current unit's QKs are done.
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(128, 128, false, false, F16);
      const uint32_t sQ = tc::smem_u32(smem + C::kQOff);
      const uint32_t sK = tc::smem_u32(smem + C::kKOff);
      tc::tma_prefetch_desc(&tmq);
      int nq = 0;  // Q copies issued; copy l goes to buffer l % NQ
      auto load_q = [&](const Unit& w, int qb) {
        ++nq;
        const int q_row0 = p.cu_q ? p.cu_q[w.b] : 0;
        const int q_b = p.cu_q ? 0 : w.b;
        unsigned char* dst = smem + C::kQOff + qb * C::kTileBytes;
        tc::mbar_arrive_expect_tx(q_full + qb, C::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tc::tma_load_4d(dst + c * 16384, &tmq, q_full + qb, c * 64, w.h, q_row0 + w.rt * 128, q_b);
      };
      bool ok = true;
      int g = 0, kk = 0;  // tiles and busy units so far
      Unit w, wn;
      int u = next_busy<INL, GTH>(p, 0, w);  // round
      if (u >= 0) load_q(w, 0);
      for (; ok && u >= 0; ++kk) {
        const int qb = kk % NQ;
        const int un = next_busy<INL, GTH>(p, u + 1, wn);
        if (!tc::mbar_wait(q_full + qb, (kk / NQ) & 1, abort_flag)) { ok = false; break; }
        for (int i = 0; i < w.count; ++i, ++g) {
          const int s = g % NSK, sb = g % NW;
          if (!tc::mbar_wait(k_full + s, (g / NSK) & 1, abort_flag)) { ok = false; break; }
          if (g >= NW && !tc::mbar_wait(s_free + sb, ((g - NW) / NW) & 1, abort_flag)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t qa = sQ + qb * C::kTileBytes, ka = sK + s * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
            tc::mma_ss(tbase + kSCol + sb * 128, tc::sdesc_sw128(qa + o, 16, 1024),
                       tc::sdesc_sw128(ka + o, 16, 1024), idS, ks > 0 ? 1u : 0u);
          }
          tc::mma_commit(s_full + sb);
          tc::mma_commit(k_empty + s);
          if (NQ == 2 && i == 0 && un >= 0) {
            // next unit's Q into the other buffer, last read by unit kk - 1
            if (kk >= 1 && !tc::mbar_wait(q_empty + (qb ^ 1), ((kk - 1) >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            load_q(wn, qb ^ 1);
          }
        }
        if (!ok) break;
        tc::mma_commit(q_empty + qb);
        if (NQ == 1 && un >= 0) {
          // one buffer: the next unit's Q once this unit's QKs have read it
          if (!tc::mbar_wait(q_empty, kk & 1, abort_flag)) {
            ok = false;
            break;
          }
          load_q(wn, 0);
        }
        u = un;
        w = wn;
      }
      if (!ok) fail(p, abort_flag, 2);
      tc::mma_commit(drained);
      tc::mbar_wait_drain(drained, 0, 200000000ull);
      if (*abort_flag) {
        // let the last Q copies land before the CTA can exit
        for (int l = nq > NQ ? nq - NQ : 0; l < nq; ++l)
          tc::mbar_wait_drain(q_full + (l % NQ), (l / NQ) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ PV issuer
    // O (+)= P[g % NW] V_g once the softmax of tile g has written P (and
    // rescaled O); the first tile of a unit overwrites O.
    if (lane == 0) {
      constexpr uint32_t idO = tc::idesc_bf16_f32(128, D, false, true, F16);
      const uint32_t sV = tc::smem_u32(smem + C::kVOff);
      bool ok = true;
      int g = 0;
      Unit w;
      for (int r = next_busy<INL, GTH>(p, 0, w); ok && r >= 0; r = next_busy<INL, GTH>(p, r + 1, w)) {
        for (int i = 0; i < w.count; ++i, ++g) {
          const int s = g % NSV, pb = g % NW;
          if (!tc::mbar_wait(p_full + pb, (g / NW) & 1, abort_flag) ||
              !tc::mbar_wait(v_full + s, (g / NSV) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t va = sV + s * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_ts(tbase + kOCol, tbase + kPCol + pb * 64 + ks * 8, tc::sdesc_sw128(va + ks * 2048, 16384, 1024),
                       idO, (i > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(p_free + pb);
          tc::mma_commit(v_empty + s);
          if (i == w.count - 1) tc::mma_commit(o_full);
        }
      }
      if (!ok) fail(p, abort_flag, 3);
      tc::mma_commit(drained + 1);
      tc::mbar_wait_drain(drained + 1, 0, 200000000ull);
    }
    __syncwarp();
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax
    // Warpgroup w takes the tiles with g % 2 == w (S and P buffer w), so one
    // warpgroup's exponentials overlap the other's loads and maxima; each
    // thread owns a whole 128-key row of its tile.  The exponent reference
    // of a row is decided tile by tile, in order: the warpgroup of tile g waits
    // for the reference posted after tile g - 1, raises it if its own maximum
    // outgrew it by more than 2^8, and posts it.  Each warpgroup keeps its own
    // row sum against the reference it last used; the two are rescaled to the
    // final reference and added at the end.  The warpgroups meet through
    // mbarriers (bounded waits), never through a named barrier, so that one
    // that gives up on a timed-out wait cannot leave the other stuck.
    const int w = NW == 2 ? (warp - 4) >> 2 : 0;
    const int wtid = tid - 128 - 128 * w;  // 0..127 within the warpgroup
    const int wq = warp & 3;               // TMEM lane quarter this warp may access
    const int row = 32 * wq + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * wq) << 16);
    float* refv = reinterpret_cast<float*>(smem + C::kRedOff);  // [2 tile parity][128]
    float* rsum = reinterpret_cast<float*>(smem + C::kSumOff);  // [2 warpgroups][128]
    unsigned char* kbuf = smem + C::kTopkOff + w * 2 * C::kTopkBuf;  // [2 buffers][lo, len, bias][128]
    constexpr int kHalfD = D / NW;  // O columns each warpgroup stores
    bool ok = true;
    int g = 0, kk = 0;  // tiles and busy units so far (all of them, both parities)
    const int nu = n_slots(p);
    // Scheduler lists: the next unit's descriptor and first list entry are
    // read a unit ahead, so that no global-memory latency sits between two
    // units.  Inline scheduling and gathered top-k units: descriptors and
    // entries are arithmetic (divisions by multiply-shift), computed where
    // they are needed, so nothing is held across the tile loop.
    constexpr bool kArith = INL || GTH;
    Unit un_next;
    if (!kArith && round_unit(0) < nu) un_next = unit_at<INL, GTH>(p, round_unit(0));
    int ent_first = 0;
    bool ent_first_ok = false;
    for (int r = 0; ok && round_unit(r) < nu; ++r) {
      const int u_next = round_unit(r + 1);  // >= nu: no next unit
      const Unit un = kArith ? unit_at<INL, GTH>(p, round_unit(r)) : un_next;
      if (!kArith && u_next < nu) un_next = unit_at<INL, GTH>(p, u_next);
      const bool pre_ok = ent_first_ok;
      ent_first_ok = false;
      if (!un.present || !un.valid) continue;
      const int b = un.b, h = un.h;
      const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
      const int off = kv_len - q_len;
      const int i = un.rt * 128 + row;
      if (un.count == 0) {
        if (w == 0 && i < q_len) write_empty_row<D>(p, b, h, i);
        continue;
      }
      int jlo_r, jhi_r;
      row_key_range(p, i, q_len, kv_len, off, jlo_r, jhi_r);
      const bool dumped = DBG && b == p.dump_b && h == p.dump_h && un.rt == p.dump_rt;
      if (DBG && dumped && w == 0 && wtid == 0) {  // the unit's list, so that entries map to key tiles
        const int64_t item = ((int64_t)b * p.Hq + h) * p.n_row_tiles + un.rt;
        p.item_count[item] = un.count;
        for (int e = 0; e < un.count; ++e) p.item_tiles[item * p.n_kt + e] = unit_entry<INL, GTH>(un, e);
      }
      const uint2* glist = GTH ? unit_glist(p, un) : nullptr;

      const float alibi_l2 = AL ? __ldg(p.alibi + h) * kLog2e : 0.f;  // ALiBi slope, log2 units
      float m_ref = -INFINITY;  // reference after the last tile seen
      float r_own = -INFINITY;  // reference this warpgroup's row sum is against
      float l = 0.f;
      // the first tile of the unit is this warpgroup's if g is of its parity
      const int it0 = (NW == 1 || (g & 1) == w) ? 0 : 1;
      // gathered keys: this thread's column entry of the warpgroup's next tile,
      // read a tile ahead so that its latency hides behind the current one
      uint2 gnext = make_uint2(0, 0);
      if (GTH && it0 < un.count) gnext = __ldg(glist + it0 * kKeysPerTile + wtid);
      int ent_cur = (kArith || !pre_ok) ? (it0 < un.count ? unit_entry<INL, GTH>(un, it0) : 0) : ent_first;
      for (int it = it0; it < un.count; it += NW) {
        const int gt = g + it;  // global index of this tile
        const int par = w;      // == gt % NW
        const int ent = kArith ? unit_entry<INL, GTH>(un, it) : ent_cur;
        if (kArith) {
        } else if (it + NW < un.count) {
          ent_cur = unit_entry<INL>(un, it + NW);
        } else if (u_next < nu && un_next.present && un_next.valid && un_next.count > 0) {
          // this warpgroup's first entry of the next unit
          const int itn = (NW == 1 || ((g + un.count) & 1) == w) ? 0 : 1;
          if (itn < un_next.count) {
            ent_first = unit_entry<INL>(un_next, itn);
            ent_first_ok = true;
          }
        }
        const int j0 = (ent >> 1) * kKeysPerTile;
        const bool part = ent & 1;
        const int kb = (gt >> 1) & 1;  // top-k staging buffer
        if (MK == FA_MASK_TOPK) {
          // column wtid of the gathered tile: the rows of this tile that keep
          // its key ([lo, hi), 8 bits each) and its bias
          const uint2 en = gnext;
          if (it + 2 < un.count) gnext = __ldg(glist + (it + 2) * kKeysPerTile + wtid);
          int* kb_lo = reinterpret_cast<int*>(kbuf + kb * C::kTopkBuf);
          const int lo = (int)((en.x >> 16) & 0xffu), hi = (int)(en.x >> 24);
          kb_lo[wtid] = lo;
          kb_lo[128 + wtid] = hi - lo;  // hi <= lo (padding) reads as no row
          reinterpret_cast<uint32_t*>(kb_lo + 256)[wtid] = en.y;
          tc::mbar_arrive(kready + 2 * w + kb);
          if (!tc::mbar_wait(kready + 2 * w + kb, (gt >> 2) & 1, abort_flag)) { ok = false; break; }
        }
        if (!tc::mbar_wait(s_full + par, (gt / NW) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        float2 x[64];
        {
          uint32_t r[4][32];
          const uint32_t sa = lane_base + kSCol + par * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) tc::tmem_ld32(sa + c * 32, r[c]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              x[c * 16 + e] = make_float2(__uint_as_float(r[c][2 * e]), __uint_as_float(r[c][2 * e + 1]));
        }
        if constexpr (DBG) {
          if (dumped) {  // raw S of this row over the tile's 128 keys
            float4* dst = reinterpret_cast<float4*>(p.dump + ((int64_t)it * 128 + row) * 128);
#pragma unroll
            for (int e4 = 0; e4 < 32; ++e4)
              dst[e4] = make_float4(x[2 * e4].x, x[2 * e4].y, x[2 * e4 + 1].x, x[2 * e4 + 1].y);
          }
        }
        tc::fence_before_sync();
        tc::mbar_arrive_relaxed(s_free + par);  // the QK NW tiles on may overwrite this S buffer
        // logits in log2 units; a FULL tile without soft-cap keeps raw scores
        // and folds the scale into the exponent below
        // Without an additive term, soft-cap or ALiBi every tile takes the
        // plain path: a PARTIAL tile first sets the raw scores of the keys
        // outside this row's range to -inf (the scale is positive, so a raw
        // -inf stays -inf through the folded scale), which keeps a single copy
        // of the exponent code in these variants.
        constexpr bool kRawMask = MK == FA_MASK_NONE && !SC && !AL;
        if (kRawMask && part) {
          // the row keeps e with clo <= e <= clo + span; a row keeping no key
          // (jhi_r < jlo_r) gets a start no e reaches
          const bool none = jhi_r < jlo_r;
          const int clo = none ? (1 << 20) : jlo_r - j0;
          const unsigned span = none ? 0u : (unsigned)(jhi_r - jlo_r);
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            x[e].x = (unsigned)(2 * e - clo) <= span ? x[e].x : -INFINITY;
            x[e].y = (unsigned)(2 * e + 1 - clo) <= span ? x[e].y : -INFINITY;
          }
        }
        const bool plain = kRawMask || (!SC && !part && !AL && MK != FA_MASK_TOPK);
        float mx;
        if (plain) {
          mx = row_max128(x) * p.scale_log2;
        } else if constexpr (MK == FA_MASK_TOPK) {
          // gathered keys: logit + bias; a PARTIAL tile also drops the keys
          // this row does not keep ((unsigned)(row - lo) >= number of rows)
          const int* kb_lo = reinterpret_cast<const int*>(kbuf + kb * C::kTopkBuf);
          const float4* kb_z = reinterpret_cast<const float4*>(kb_lo + 256);
          const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float4 z4 = kb_z[c];
            float2 a = x[2 * c], bq = x[2 * c + 1];
            if (SC) {
              a = make_float2(softcap_log2(a.x * p.scale, p.softcap, p.inv_softcap) + z4.x,
                              softcap_log2(a.y * p.scale, p.softcap, p.inv_softcap) + z4.y);
              bq = make_float2(softcap_log2(bq.x * p.scale, p.softcap, p.inv_softcap) + z4.z,
                               softcap_log2(bq.y * p.scale, p.softcap, p.inv_softcap) + z4.w);
            } else {
              a = fma2(a, sl2, make_float2(z4.x, z4.y));
              bq = fma2(bq, sl2, make_float2(z4.z, z4.w));
            }
            if (part) {
              const int4 lo4 = reinterpret_cast<const int4*>(kb_lo)[c];
              const int4 n4 = reinterpret_cast<const int4*>(kb_lo + 128)[c];
              a.x = (unsigned)(row - lo4.x) < (unsigned)n4.x ? a.x : -INFINITY;
              a.y = (unsigned)(row - lo4.y) < (unsigned)n4.y ? a.y : -INFINITY;
              bq.x = (unsigned)(row - lo4.z) < (unsigned)n4.z ? bq.x : -INFINITY;
              bq.y = (unsigned)(row - lo4.w) < (unsigned)n4.w ? bq.y : -INFINITY;
            }
            x[2 * c] = a;
            x[2 * c + 1] = bq;
          }
          mx = row_max128(x);
        } else {
          const int clo = jlo_r - j0, chi = jhi_r - j0;
          const float* mrow = nullptr;
          if (MK == FA_MASK_DENSE && i < q_len)
            mrow = p.mask + (int64_t)(p.m_nb > 1 ? b : 0) * p.m_sb + (int64_t)(p.m_nh > 1 ? h : 0) * p.m_sh +
                   (int64_t)i * p.m_sq + (int64_t)j0 * p.m_sk;
#pragma unroll
          for (int e = 0; e < 128; ++e) {
            float v = (e & 1) ? x[e >> 1].y : x[e >> 1].x;
            if (SC) {
              v = softcap_log2(v * p.scale, p.softcap, p.inv_softcap);
            } else {
              v = v * p.scale_log2;
            }
            if (AL) v -= alibi_l2 * (float)abs(i + off - (j0 + e));
            bool keep = !part || (e >= clo && e <= chi);
            if (MK == FA_MASK_DENSE && part) {
              if (keep) v += __ldg(mrow + (int64_t)e * p.m_sk) * kLog2e;
            }
            v = keep ? v : -INFINITY;
            if (e & 1) x[e >> 1].y = v; else x[e >> 1].x = v;
          }
          mx = row_max128(x);
        }
        // the reference after tile gt - 1 (with two warpgroups every tile's
        // reference is posted, also across units, so that they stay in step)
        if (NW == 2 && gt >= 1 && !tc::mbar_wait(refb + (par ^ 1), ((gt - 1) >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const float m_prev = (it == 0) ? -INFINITY : (NW == 2 ? refv[(par ^ 1) * 128 + row] : m_ref);
        // raise the exponent reference only when the row max outgrew it by 2^8
        const bool upd = mx > m_prev + kRescaleLog2;
        m_ref = upd ? mx : m_prev;
        if (NW == 2) {
          refv[par * 128 + row] = m_ref;
          tc::mbar_arrive(refb + par);
        }
        if (it != 0 && __any_sync(0xffffffffu, upd && m_prev != -INFINITY)) {
          // O holds the PV of tile gt - 1 (against m_prev) once that PV is done
          if (!tc::mbar_wait(p_free + (gt - 1) % NW, ((gt - 1) / NW) & 1, abort_flag)) { ok = false; break; }
          tc::fence_after_sync();
          const float f = (upd && m_prev != -INFINITY) ? fast_exp2(m_prev - m_ref) : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            const uint32_t a = lane_base + kOCol + c * 32;
            tc::tmem_ld32(a, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
            tc::tmem_st32(a, r);
          }
        }
        if (r_own != m_ref) {
          l = (r_own == -INFINITY) ? 0.f : l * fast_exp2(r_own - m_ref);
          r_own = m_ref;
        }
        const float eref = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 ner = make_float2(-eref, -eref);
        float2 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
        // P = exp2(x - ref) packed to input-type pairs in registers: one packed FMA
        // (FULL: scale folded in) or add per pair
        uint32_t pk[4][16];
        if (plain) {
          const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = fma2(x[c * 16 + e], sl2, ner);
              const float2 pe = make_float2(fast_exp2(v.x), fast_exp2(v.y));
              acc[e & 3] = add2(acc[e & 3], pe);
              pk[c][e] = pack2<F16>(pe.x, pe.y);
            }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 v = add2(x[c * 16 + e], ner);
              const float2 pe = make_float2(fast_exp2(v.x), fast_exp2(v.y));
              acc[e & 3] = add2(acc[e & 3], pe);
              pk[c][e] = pack2<F16>(pe.x, pe.y);
            }
        }
        if constexpr (DBG) {
          if (dumped) {  // P as rounded for PV, and the reference
            float* dp = p.dump + ((int64_t)(p.n_kt + it) * 128 + row) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float lo, hi;
                if constexpr (F16) {
                  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pk[c][e]));
                  lo = f.x;
                  hi = f.y;
                } else {
                  lo = __uint_as_float(pk[c][e] << 16);
                  hi = __uint_as_float(pk[c][e] & 0xffff0000u);
                }
                dp[2 * (c * 16 + e)] = lo;
                dp[2 * (c * 16 + e) + 1] = hi;
              }
            p.dump[(int64_t)2 * p.n_kt * 128 * 128 + (int64_t)it * 128 + row] = eref;
          }
        }
        // this P buffer is free once the PV NW tiles back is done
        if (gt >= NW && !tc::mbar_wait(p_free + par, ((gt - NW) / NW) & 1, abort_flag)) { ok = false; break; }
        const uint32_t pa = lane_base + kPCol + par * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_st16(pa + c * 16, pk[c]);
        acc[0] = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
        l += acc[0].x + acc[0].y;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive_relaxed(p_full + par);
      }
      if (!ok) break;
      // ---- epilogue: both warpgroups' row sums against the final reference
      const int gl = g + un.count - 1;  // the unit's last tile
      g += un.count;
      if (NW == 2 && (gl & 1) != w) {
        if (!tc::mbar_wait(refb + (gl & 1), (gl >> 1) & 1, abort_flag)) { ok = false; break; }
        m_ref = refv[(gl & 1) * 128 + row];
      }
      // this warpgroup's O columns are read out of TMEM before its row sum is
      // posted: the next unit's first PV overwrites O, and its P comes from a
      // warpgroup that has passed the row-sum barrier (with one warpgroup:
      // from this one, after the read), so every O read is ordered before
      // that PV
      if (!tc::mbar_wait(o_full, kk & 1, abort_flag)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t ro[kHalfD / 32][32];
#pragma unroll
      for (int c = 0; c < kHalfD / 32; ++c) tc::tmem_ld32(lane_base + kOCol + w * kHalfD + c * 32, ro[c]);
      float lt;
      if constexpr (NW == 2) {
        rsum[w * 128 + row] = (r_own == m_ref || r_own == -INFINITY) ? l : l * fast_exp2(r_own - m_ref);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        tc::mbar_arrive(sumx);
        if (!tc::mbar_wait(sumx, kk & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        lt = rsum[row] + rsum[128 + row];
      } else {
        // one warpgroup: its row sum is against the last reference already
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        lt = l;
      }
      const bool empty = !(lt > 0.f);
      const float inv = empty ? 0.f : 1.f / lt;
      const float lse2 = empty ? -INFINITY : m_ref + __log2f(lt);  // log2-sum-exp of the row
      const int64_t qbase = p.cu_q ? (int64_t)p.cu_q[b] : 0;
      uint16_t* obase = p.o + (p.cu_q ? 0 : (int64_t)b * p.o_sb) + (int64_t)h * p.o_sh;
      // the piece this slot holds, worked out again here rather than kept
      // live through the tile loop (a unit of fewer than two tiles is whole)
      constexpr bool kTail = INL && NW == 2;  // compiled into the d = 128 variants only
      int tu = 0;
      int piece = kTail ? tail_piece<INL>(p, round_unit(r), tu) : 0;
      if (piece == 1 && unit_of<INL, GTH>(p, p.tail_round * (int)gridDim.x + tu).count < 2) piece = 0;
      if (kTail && piece != 0) {
        // A piece of a split tail unit stores its normalised O and
        // log2-sum-exp, per warpgroup half of the columns, [column][row] so
        // that a warp's stores and loads are contiguous.  The piece whose
        // warpgroup arrives second on the unit's 2-bit count (which it
        // returns to zero) merges the two from memory and writes the rows:
        // O = (O1 2^L1 + O2 2^L2) / (2^L1 + 2^L2), L = log2(2^L1 + 2^L2).
        constexpr int kSlot = 128 * D + 256;
        float* mine = p.tail_part + (int64_t)(2 * tu + piece - 1) * kSlot;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) __stcg(mine + (w * kHalfD + c * 32 + e) * 128 + row, __uint_as_float(ro[c][e]) * inv);
        __stcg(mine + 128 * D + w * 128 + row, lse2);
        __threadfence();
        tc::mbar_arrive(tdone + w);
        if (wtid == 0) {
          int dec = 2;
          if (tc::mbar_wait(tdone + w, 0, abort_flag)) {
            __threadfence();
            const int f = 2 * (2 * tu + w);
            uint32_t* word = p.tail_flags + (f >> 5);
            const uint32_t old = atomicAdd(word, 1u << (f & 31));
            dec = ((old >> (f & 31)) & 3u) == 1u ? 1 : 0;
            if (dec == 1) atomicSub(word, 2u << (f & 31));
          }
          tsec[w] = dec;
          tc::mbar_arrive(tflag + w);
        }
        if (!tc::mbar_wait(tflag + w, 0, abort_flag) || tsec[w] == 2) { ok = false; break; }
        if (tsec[w] == 1) {
          __threadfence();
          const float* oth = p.tail_part + (int64_t)(2 * tu + 2 - piece) * kSlot;
          const float lo = __ldcg(oth + 128 * D + w * 128 + row);
          const float mx = fmaxf(lse2, lo);
          float fa = 0.f, fb = 0.f;  // weights of this piece's rows and the other's
          float lm = -INFINITY;
          if (mx != -INFINITY) {
            const float ea = fast_exp2(lse2 - mx), eb = fast_exp2(lo - mx);
            const float sum = ea + eb;
            fa = ea / sum;
            fb = eb / sum;
            lm = mx + __log2f(sum);
          }
          if (i < q_len) {
            uint16_t* orow = obase + (qbase + i) * p.o_ss + w * kHalfD;
            // eight columns per step: a wider step (more loads in flight)
            // measured slower, as the registers it takes cost the tile loop
#pragma unroll 1
            for (int c0 = 0; c0 < kHalfD; c0 += 8) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                v[e] = __ldcg(mine + (w * kHalfD + c0 + e) * 128 + row) * fa +
                       __ldcg(oth + (w * kHalfD + c0 + e) * 128 + row) * fb;
              uint4 o4;
              o4.x = pack2<F16>(v[0], v[1]);
              o4.y = pack2<F16>(v[2], v[3]);
              o4.z = pack2<F16>(v[4], v[5]);
              o4.w = pack2<F16>(v[6], v[7]);
              *reinterpret_cast<uint4*>(orow + c0) = o4;
            }
            if (w == 0) {
              float* lptr = p.lse + (p.cu_q ? 0 : (int64_t)b * p.lse_sb) + (int64_t)h * p.lse_sh + (qbase + i) * p.lse_ss;
              *lptr = lm * kLn2;
            }
          }
        }
      } else {
        // O / l through a warp-private staging tile: a thread packs its own row,
        // then each store instruction writes 64 contiguous bytes of 8 rows
        uint4* stg = reinterpret_cast<uint4*>(smem + C::kStageOff + (warp - 4) * 2048);  // [32 rows][4]
        const int row0 = un.rt * 128 + 32 * wq;  // first row of this warp
        // whole 32-row chunks inside the sequence leave by TMA store
        const bool tma_rows = o_tma && row0 + 32 <= q_len;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          const uint32_t* r = ro[c];
          // the staging tile is free once the previous TMA store has read it
          if (lane == 0) tc::bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 o4;
            o4.x = pack2<F16>(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
            o4.y = pack2<F16>(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
            o4.z = pack2<F16>(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
            o4.w = pack2<F16>(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
            stg[lane * 4 + (v4 ^ ((lane >> 1) & 3))] = o4;  // swizzled: 4 wavefronts
          }
          if (tma_rows) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_4d(&tmo, stg, w * kHalfD + c * 32, h, (int)(qbase + row0), p.cu_q ? 0 : b);
              tc::bulk_commit();
            }
          } else {
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rr = 8 * k + (lane >> 2), q = lane & 3;
              const uint4 o4 = stg[rr * 4 + (q ^ ((rr >> 1) & 3))];
              if (row0 + rr < q_len)
                *reinterpret_cast<uint4*>(obase + (qbase + row0 + rr) * p.o_ss + w * kHalfD + c * 32 + 8 * q) = o4;
            }
            __syncwarp();
          }
        }
        if (w == 0 && i < q_len) {
          float* lptr = p.lse + (p.cu_q ? 0 : (int64_t)b * p.lse_sb) + (int64_t)h * p.lse_sh + (qbase + i) * p.lse_ss;
          *lptr = lse2 * kLn2;
        }
      }
      ++kk;
    }
    if (!ok) fail(p, abort_flag, 4 + w);
    // output stores complete before the CTA exits
    if (lane == 0) tc::bulk_wait_all();
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tbase, C::kCols);
  if (INL && blockIdx.x == 0 && warp == 2) inline_sched_stats(p);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 4-D map {d, heads, rows, batch} over a bshd (or packed thd) bf16 / fp16 tensor,
// box {64, 1, 128, 1}, 128-byte swizzle; rows beyond the tensor read as 0.
bool encode_bshd(CUtensorMap* m, const void* base, int d, int heads, int64_t rows, int batch, int64_t s_h,
                 int64_t s_row, int64_t s_b, bool f16) {
  return encode_4d_bf16(m, base, d, heads, rows, batch, s_h, s_row, s_b, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, f16);
}

// 4-D map over the output for the epilogue's TMA stores: box {32, 1, 32,
// 1} (32 columns x 32 rows), 64-byte swizzle (the staging layout).
bool encode_out(CUtensorMap* m, void* base, int d, int heads, int64_t rows, int batch, int64_t s_h, int64_t s_row,
                int64_t s_b, bool f16) {
  return encode_4d_bf16(m, base, d, heads, rows, batch, s_h, s_row, s_b, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, f16);
}

// SM count of the current device (cached per device; safe to call from
// several host threads).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  const int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return 1;
  }
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

template <int D, int MK, bool SC, bool AL, bool F16, bool DBG = false>
cudaError_t launch_prefill_v(const Params& p, cudaStream_t st, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, const CUtensorMap& mo, int o_tma, int grid,
                             cudaEvent_t ev_begin) {
  // setmaxnreg.inc would wait forever if the block were launched with fewer
  // registers than the split assumes: launch only when the build matches.
  static std::atomic<int> launch_regs{-1};
  int regs = launch_regs.load(std::memory_order_relaxed);
  if (regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_kernel<D, MK, SC, AL, F16, DBG>);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
    launch_regs.store(regs, std::memory_order_relaxed);
  }
  if (regs != prefill_launch_regs(D, MK)) return cudaErrorInvalidConfiguration;
  using C = PCfg<D, MK == FA_MASK_TOPK>;
  cudaError_t e = ensure_smem_attr<prefill_kernel<D, MK, SC, AL, F16, DBG>>(C::kSmem);
  if (e != cudaSuccess) return e;
  if (ev_begin && (e = cudaEventRecord(ev_begin, st)) != cudaSuccess) return e;
  prefill_kernel<D, MK, SC, AL, F16, DBG><<<(unsigned)grid, prefill_threads(D, MK), C::kSmem, st>>>(p, mq, mk, mv, mo, o_tma);
  return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_prefill_d(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  CUtensorMap mq, mk, mv;
  const bool vq = p.cu_q != nullptr, vk = p.cu_k != nullptr;
  // extents of 1 get a harmless stride (the stride of the next-inner dimension)
  const int64_t q_rows = vq ? p.tot_q : p.Sq, k_rows = vk ? p.tot_k : p.Sk;
  const int qb = vq ? 1 : p.n_seq, kb = vk ? 1 : p.n_seq;
  const int64_t q_sb = (qb == 1 || p.q_sb == 0) ? p.q_ss : p.q_sb;
  const int64_t k_sb = (kb == 1 || p.k_sb == 0) ? p.k_ss : p.k_sb;
  const int64_t v_sb = (kb == 1 || p.v_sb == 0) ? p.v_ss : p.v_sb;
  const int64_t o_sb = (qb == 1 || p.o_sb == 0) ? p.o_ss : p.o_sb;
  CUtensorMap mo;
  // without a valid map (unusual strides) the epilogue uses plain stores
  const int o_tma = encode_out(&mo, p.o, D, p.Hq, q_rows, qb, p.o_sh, p.o_ss, o_sb, F16) ? 1 : 0;
  if (!o_tma) memset(&mo, 0, sizeof(mo));
  if (!encode_bshd(&mq, p.q, D, p.Hq, q_rows, qb, p.q_sh, p.q_ss, q_sb, F16)) return cudaErrorInvalidValue;
  if (p.mask_kind == FA_MASK_TOPK) {
    // gathered keys: 2-D views with row b * Sk + j = key j of sequence b (all
    // heads of a key side by side; the planner checked that the layout is one)
    if (vk) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)p.n_seq * p.Sk;
    if (!encode_rows_bf16(&mk, p.k, (int64_t)(p.Hkv - 1) * p.k_sh + D, rows, p.k_ss, 64, F16) ||
        !encode_rows_bf16(&mv, p.v, (int64_t)(p.Hkv - 1) * p.v_sh + D, rows, p.v_ss, 64, F16))
      return cudaErrorInvalidValue;
  } else if (!encode_bshd(&mk, p.k, D, p.Hkv, k_rows, kb, p.k_sh, p.k_ss, k_sb, F16) ||
             !encode_bshd(&mv, p.v, D, p.Hkv, k_rows, kb, p.v_sh, p.v_ss, v_sb, F16)) {
    return cudaErrorInvalidValue;
  }
  // the planner's grid (plan_prefill_grid)
  const int64_t units = (int64_t)p.n_row_tiles * p.n_seq * p.Hq;
  if (units <= 0) return ev_begin ? cudaEventRecord(ev_begin, st) : cudaSuccess;
  if (units > INT_MAX || p.prefill_grid <= 0) return cudaErrorInvalidValue;
  if (p.tail_units > 0 && (p.mask_kind != FA_MASK_NONE || p.dump)) return cudaErrorInvalidValue;
  const int grid = p.prefill_grid;
  const bool sc = p.softcap > 0.f;
  // the kernels schedule inline exactly for the mask-free variants
  if ((p.sched_inline != 0) != (p.mask_kind == FA_MASK_NONE)) return cudaErrorInvalidValue;
  if (p.dump) {  // the debug instantiations: bf16, no additive term (the planner checks)
    if constexpr (F16) {
      return cudaErrorInvalidValue;
    } else {
      if (p.alibi || p.mask_kind != FA_MASK_NONE) return cudaErrorInvalidValue;
      return sc ? launch_prefill_v<D, FA_MASK_NONE, true, false, F16, true>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_NONE, false, false, F16, true>(p, st, mq, mk, mv, mo, o_tma, grid,
                                                                              ev_begin);
    }
  }
  if (p.alibi) {  // the planner allows ALiBi in prefill without a mask or with a dense one
    if (p.mask_kind == FA_MASK_TOPK) return cudaErrorInvalidValue;
    if (p.mask_kind == FA_MASK_DENSE)
      return sc ? launch_prefill_v<D, FA_MASK_DENSE, true, true, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_DENSE, false, true, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin);
    return sc ? launch_prefill_v<D, FA_MASK_NONE, true, true, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
              : launch_prefill_v<D, FA_MASK_NONE, false, true, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin);
  }
  switch (p.mask_kind) {
    case FA_MASK_DENSE:
      return sc ? launch_prefill_v<D, FA_MASK_DENSE, true, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_DENSE, false, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin);
    case FA_MASK_TOPK:
      return sc ? launch_prefill_v<D, FA_MASK_TOPK, true, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_TOPK, false, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin);
    default:
      return sc ? launch_prefill_v<D, FA_MASK_NONE, true, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin)
                : launch_prefill_v<D, FA_MASK_NONE, false, false, F16>(p, st, mq, mk, mv, mo, o_tma, grid, ev_begin);
  }
}

}  // namespace

// The fp16 instantiations are compiled in their own translation unit
// (prefill_f16.cu includes this file with MFA_PREFILL_F16_UNIT defined), so
// that the two element types build in parallel.
#ifndef MFA_PREFILL_F16_UNIT
void plan_prefill_grid(Params& p) {
  // one CTA per SM (two at d = 64 without top-k; persistent), never more
  // CTAs than work units
  const int64_t units = (int64_t)p.n_row_tiles * p.n_seq * p.Hq;
  p.prefill_grid = p.tail_round = p.tail_units = 0;
  if (units <= 0 || units > INT_MAX) return;
  const int64_t slots = (int64_t)sm_count() * prefill_ctas_per_sm(p.d, p.mask_kind);
  const int grid = (int)(units < slots ? units : slots);
  p.prefill_grid = grid;
  // Without a mask the units of a launch have nearly equal lengths (a causal
  // launch over past keys) or fall in length from round to round; a last
  // round that fills at most half the grid would leave most SMs idle while
  // it runs, so its units are cut in two over their key tiles.  Each piece
  // pays a unit's fixed costs and its rows a store, a load and a merge: the
  // split is taken when every unit of that round has kTailMinTiles key tiles
  // or more, which the host knows for sequences of one length (the last
  // round holds the smallest row tiles: those of units rounds * grid ..
  // units - 1).
  constexpr int kTailMinTiles = 4;
  const int64_t rounds = units / grid, left = units - rounds * grid;
  constexpr int64_t kFlagBits = (int64_t)(kWsHeadBytes - kTailFlagsOff) * 8;
  // (d = 64 launches run two CTAs per SM, whose units' epilogues already
  // overlap: no split there)
  if (p.mask_kind != FA_MASK_NONE || p.d != 128 || p.cu_q || p.cu_k || p.cache_len || rounds < 1 || left <= 0 ||
      2 * left > grid || 4 * left > kFlagBits)
    return;
  const int64_t per_rt = (int64_t)p.n_seq * p.Hq;
  const int rt_hi = p.n_row_tiles - 1 - (int)(rounds * grid / per_rt), rt_lo = p.n_row_tiles - 1 - (int)((units - 1) / per_rt);
  const bool no_skip = (p.debug_flags & FA_DEBUG_NO_SKIP) != 0;
  for (int rt = rt_lo; rt <= rt_hi; ++rt) {
    // the unit's key range under the pair rules, as the kernel derives it
    const int64_t i0 = (int64_t)rt * 128, i1 = std::min<int64_t>(i0 + 127, p.Sq - 1), off = (int64_t)p.Sk - p.Sq;
    int64_t jlo = 0, jhi = p.Sk - 1;
    if (!no_skip) {
      if (p.causal) jhi = std::min(jhi, i1 + off);
      if (p.wl >= 0) jlo = std::max(jlo, i0 + off - p.wl);
      if (p.wr >= 0) jhi = std::min(jhi, i1 + off + p.wr);
    }
    if (jlo > jhi || jhi / kKeysPerTile - jlo / kKeysPerTile + 1 < kTailMinTiles) return;
  }
  p.tail_round = (int32_t)rounds;
  p.tail_units = (int32_t)left;
}

cudaError_t launch_prefill(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  if (p.n_items <= 0) return ev_begin ? cudaEventRecord(ev_begin, st) : cudaSuccess;
  if (p.f16) return launch_prefill_f16(p, st, ev_begin);
  return p.d == 64 ? launch_prefill_d<64, false>(p, st, ev_begin) : launch_prefill_d<128, false>(p, st, ev_begin);
}
#else
cudaError_t launch_prefill_f16(const Params& p, cudaStream_t st, cudaEvent_t ev_begin) {
  return p.d == 64 ? launch_prefill_d<64, true>(p, st, ev_begin) : launch_prefill_d<128, true>(p, st, ev_begin);
}
#endif

}  // namespace mfa
