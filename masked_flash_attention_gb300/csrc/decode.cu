// decode.cu -- split-KV attention for few query rows per K/V head (decode,
// speculative decode, short chunks), plus the split combine pass.
//
// One CTA = one item (sequence, K/V head, 8 packed rows) x one split of its
// scheduled key tiles.  The packed rows are the query heads of the K/V head's
// group times the query positions, so a group shares every K/V byte it reads
// (grouped-query heads without K/V expansion, InfiniTrain pull request 193
// "Transformer 接入").  The split's keys are cut into 16-key chunks dealt out
// round-robin to the 4 warps; every warp streams its own chunks through a
// private 3-stage shared-memory ring with 16-byte cp.async copies (each
// instruction of a warp covers two whole K or V rows, so the copies are fully
// coalesced), through the paged block_table when there is one (vLLM pull
// request 11277's flash_attn_varlen_func `block_table`; one page lookup per
// chunk when the page size is a multiple of 16).  Warps never wait for each
// other until the end.  S^T = K Q^T and O^T += V^T P^T run on mma.sync
// m16n8k16 (bf16 in, fp32 accumulate) with keys / head-dim on M and the 8 query
// rows on N, so a group of 4 q-heads wastes half of N instead of 3/4 of M;
// 8 rows are far too few for a 128-row tcgen05 tile.  The
// running softmax is guarded so that a fully masked chunk never produces NaN
// (ExecuTorch pull request 10466 "Summary").
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fa_device.cuh"
#include "host_util.h"
#include "mma_sync.cuh"
#include "tc_sm103.cuh"

namespace mfa {

namespace {

constexpr int kChunkKeys = 16;   // keys per warp stage
constexpr int kWarpStages = 3;   // stages in flight per warp
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

template <int D>
struct DecodeSmem {
  static constexpr int kChunks = D / 8;                        // 16-byte chunks per row
  static constexpr int kKvBytes = kChunkKeys * D * 2;          // K or V of one warp stage
  static constexpr int kStageBytes = 2 * kKvBytes;
  static constexpr int kWarpBytes = kWarpStages * kStageBytes;
  static constexpr int kQBytes = kDecodeRows * D * 2;
  static constexpr int kBarOff = kWarps * kWarpBytes + kQBytes;  // TMA mode: [warp][stage] mbarriers + abort flag
  static constexpr int kTotal = kBarOff + kWarps * kWarpStages * 8 + 16 + 1024;  // + alignment slack
  static_assert(kWarps * kDecodeRows * D * 4 <= kWarps * kWarpBytes, "merge buffer must fit");
  static_assert(2 * kWarps * kDecodeRows * 4 <= kQBytes, "warp statistics must fit over Q");
};

// Address of key/value row j (head g) of sequence b.
__device__ __forceinline__ const uint16_t* kv_row(const Params& p, const uint16_t* base, int64_t sb,
                                                  int64_t ss, int64_t sh, int b, int g, int j) {
  if (p.block_table) {
    int pg = __ldg(p.block_table + (int64_t)b * p.bt_stride + j / p.page_size);
    if ((unsigned)pg >= (unsigned)p.num_pages) {
      record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)pg);
      pg = 0;
    }
    return base + (int64_t)pg * sb + (int64_t)(j % p.page_size) * ss + (int64_t)g * sh;
  }
  if (p.cu_k) return base + (int64_t)(p.cu_k[b] + j) * ss + (int64_t)g * sh;
  return base + (int64_t)b * sb + (int64_t)j * ss + (int64_t)g * sh;
}

// Key/value row j (head g) of sequence b, cached keys first: rows j >= lc
// are the sequence's active rows j - lc in k_new / v_new (laid out like q).
__device__ __forceinline__ const uint16_t* kv_src_row(const Params& p, bool is_v, int b, int g, int j, int lc) {
  if (j >= lc) {
    const int64_t r = (p.cu_q ? (int64_t)p.cu_q[b] : 0) + (j - lc);
    return is_v ? p.v_new + (p.cu_q ? 0 : (int64_t)b * p.vn_sb) + r * p.vn_ss + (int64_t)g * p.vn_sh
                : p.k_new + (p.cu_q ? 0 : (int64_t)b * p.kn_sb) + r * p.kn_ss + (int64_t)g * p.kn_sh;
  }
  return is_v ? kv_row(p, p.v, p.v_sb, p.v_ss, p.v_sh, b, g, j) : kv_row(p, p.k, p.k_sb, p.k_ss, p.k_sh, b, g, j);
}

// Append (two-source form): the active rows of sequence b, head g, are copied
// into the cache at rows lc .. lc + q_len - 1 by one CTA per (sequence, K/V
// head).  The scheduler has checked lc + q_len against the cache capacity; a
// bad page index is recorded and its rows are not written.
template <int D>
__device__ void append_active(const Params& p, int b, int g, int lc, int q_len, int tid, int nthreads) {
  constexpr int kPieces = D / 8;
  for (int idx = tid; idx < q_len * kPieces; idx += nthreads) {
    const int t = idx / kPieces, c = idx % kPieces;
    const int j = lc + t;
    int64_t ko, vo;
    if (p.block_table) {
      const int pg = __ldg(p.block_table + (int64_t)b * p.bt_stride + j / p.page_size);
      if ((unsigned)pg >= (unsigned)p.num_pages) {
        record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)pg);
        continue;
      }
      ko = (int64_t)pg * p.k_sb + (int64_t)(j % p.page_size) * p.k_ss;
      vo = (int64_t)pg * p.v_sb + (int64_t)(j % p.page_size) * p.v_ss;
    } else {
      ko = (int64_t)b * p.k_sb + (int64_t)j * p.k_ss;
      vo = (int64_t)b * p.v_sb + (int64_t)j * p.v_ss;
    }
    ko += (int64_t)g * p.k_sh + c * 8;
    vo += (int64_t)g * p.v_sh + c * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(kv_src_row(p, false, b, g, j, lc) + c * 8);
    const uint4 vv = *reinterpret_cast<const uint4*>(kv_src_row(p, true, b, g, j, lc) + c * 8);
    *reinterpret_cast<uint4*>(const_cast<uint16_t*>(p.k) + ko) = kv;
    *reinterpret_cast<uint4*>(const_cast<uint16_t*>(p.v) + vo) = vv;
  }
}

struct ItemGeo {
  int b, g, rt, q_len, kv_len, off, i0, i1, jlo, jhi;
  int lc;  // keys held in the cache (two-source form), else kv_len
};

template <bool KV2 = true>
__device__ __forceinline__ ItemGeo item_geo(const Params& p, int64_t item) {
  ItemGeo t;
  t.rt = (int)(item % p.n_row_tiles);
  int64_t r = item / p.n_row_tiles;
  t.g = (int)(r % p.n_heads_sched);
  t.b = (int)(r / p.n_heads_sched);
  t.q_len = seq_qlen(p, t.b);
  t.kv_len = seq_klen(p, t.b);
  t.off = t.kv_len - t.q_len;
  t.lc = (KV2 && p.cache_len) ? __ldg(p.cache_len + t.b) : t.kv_len;
  tile_rows(p, t.rt, t.i0, t.i1);
  t.i1 = min(t.i1, t.q_len - 1);
  key_range(p, t.i0, t.i1, t.off, t.kv_len, t.jlo, t.jhi);
  if (p.debug_flags & FA_DEBUG_NO_SKIP) { t.jlo = 0; t.jhi = t.kv_len - 1; }
  return t;
}

// Output row pointers / LSE index for packed row P of an item.
__device__ __forceinline__ void out_ptrs(const Params& p, const ItemGeo& t, int P, uint16_t*& optr,
                                         float*& lptr, bool& valid) {
  int qi = P / p.G, h = t.g * p.G + P % p.G;
  valid = qi < t.q_len;
  int64_t qrow = p.cu_q ? (int64_t)p.cu_q[t.b] + qi : (int64_t)qi;
  int64_t bo = p.cu_q ? 0 : (int64_t)t.b;
  optr = p.o + bo * p.o_sb + qrow * p.o_ss + (int64_t)h * p.o_sh;
  lptr = p.lse + bo * p.lse_sb + (int64_t)h * p.lse_sh + qrow * p.lse_ss;
}

// byte offset of (row, 16-byte column chunk cc) in a TMA-written chunk: two
// 64-column halves of 16 rows x 128 bytes, 128-byte swizzle
__device__ __forceinline__ uint32_t swz_tma(int row, int cc) {
  return (uint32_t)((cc >> 3) * (kChunkKeys * 128) + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
}

// Zero rows [first, 16) of a TMA-layout V stage (all lanes of the warp; kept
// out of line: it runs on a sequence's last chunk only).
template <int D>
__device__ __noinline__ void zero_rows_from(uint32_t sV, int first, int lane) {
  constexpr int kPieces = D / 8;
  for (int idx = lane; idx < kChunkKeys * kPieces; idx += 32) {
    const int r = idx / kPieces, c = idx % kPieces;
    if (r >= first) asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(sV + swz_tma(r, c)), "r"(0));
  }
  __syncwarp();
}

// Merge the 4 consumer warps' (m, l, O) and write the item's rows, or this
// split's partial rows when the item has several splits.  Run by the 128
// consumer threads only (thread ids 0..127), which meet on named barrier 1;
// `smem` (16 KB at d = 128) is free for the merge buffer, `red_m` points to
// 2 x 4 x 8 floats that are not part of it.
template <int D, bool F16>
__device__ __forceinline__ void decode_finish(const Params& p, const ItemGeo& geo, int64_t item, int split,
                                              bool single, unsigned char* smem, float* red_m, int tid,
                                              float (&m_run)[2], float (&l_run)[2], float (&o_acc)[D / 16][4]) {
  const int warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;
  // ---- merge the 4 warps' (m, l, O) ----
  float* red_l = red_m + kWarps * kDecodeRows;
  float* obuf = reinterpret_cast<float*>(smem);  // [4][8][D]
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 4);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 8);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 16);
  }
  if (g8 == 0) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      red_m[warp * kDecodeRows + 2 * c4 + rr] = m_run[rr];
      red_l[warp * kDecodeRows + 2 * c4 + rr] = l_run[rr];
    }
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  float f_own[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = 2 * c4 + rr;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * kDecodeRows + row]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    f_own[rr] = fast_exp2(m_run[rr] - Mref);
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    float* ow = obuf + (warp * kDecodeRows) * D;
    ow[(2 * c4) * D + 16 * mt + g8] = o_acc[mt][0] * f_own[0];
    ow[(2 * c4 + 1) * D + 16 * mt + g8] = o_acc[mt][1] * f_own[1];
    ow[(2 * c4) * D + 16 * mt + g8 + 8] = o_acc[mt][2] * f_own[0];
    ow[(2 * c4 + 1) * D + 16 * mt + g8 + 8] = o_acc[mt][3] * f_own[1];
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  // each thread: one row, D/16 consecutive columns
  {
    constexpr int kCols = D / 16;
    const int row = tid >> 4;  // 8 rows x 16 threads
    const int c0 = (tid & 15) * kCols;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * kDecodeRows + row]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      L += red_l[w * kDecodeRows + row] * fast_exp2(red_m[w * kDecodeRows + row] - Mref);
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
    const float lse_val = empty ? -INFINITY : (Mref + __log2f(L)) * kLn2;
    float vals[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc += obuf[(w * kDecodeRows + row) * D + c0 + c];
      vals[c] = acc * inv;
    }
    const int P = geo.rt * kDecodeRows + row;
    if (single) {
      uint16_t* optr; float* lptr; bool valid;
      out_ptrs(p, geo, P, optr, lptr, valid);
      if (valid) {
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          uint2 pk;
          pk.x = pack_bf16<F16>(vals[c + 0], vals[c + 1]);
          pk.y = pack_bf16<F16>(vals[c + 2], vals[c + 3]);
          *reinterpret_cast<uint2*>(optr + c0 + c) = pk;
        }
        if ((tid & 15) == 0) *lptr = lse_val;
      }
    } else {
      int64_t slot = (item * p.n_splits + split) * kDecodeRows + row;
      float* po = p.part_o + slot * D + c0;
#pragma unroll
      for (int c = 0; c < kCols; c += 4)
        *reinterpret_cast<float4*>(po + c) = make_float4(vals[c], vals[c + 1], vals[c + 2], vals[c + 3]);
      if ((tid & 15) == 0) p.part_lse[slot] = lse_val;
    }
  }
}

// TMA: K/V chunks arrive by TMA tensor copies (a 16-row box of one K/V head:
// one page, or 16 consecutive rows), issued by lane 0 of the warp that owns
// the ring and tracked by one mbarrier per stage; otherwise by 16-byte
// cp.async from all lanes (any layout).
template <int D, bool TMA, bool F16, bool KV2>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const Params p, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using S = DecodeSmem<D>;
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned base: the TMA copies use the 128-byte swizzle
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // splits slowest: every item's first split is dispatched before any second
  // one, so the grid ends on the last splits of the longest sequences (partial
  // or empty) rather than on the full-length splits of the last items
  const int64_t cta = blockIdx.x;
  const int split = (int)(cta / p.n_items);
  const int64_t item = cta - (int64_t)split * p.n_items;
  const int count = p.item_count[item];
  if (count < 0) return;  // sequence rejected by the scheduler's length checks
  const int t_begin = split * p.tiles_per_split;
  // an item with nothing scheduled still owes its rows O = 0, LSE = -inf
  if (t_begin >= count && !(split == 0 && count == 0)) return;
  const int t_end = min(count, t_begin + p.tiles_per_split);
  const bool single = count <= p.tiles_per_split;
  const ItemGeo geo = item_geo<KV2>(p, item);
  const int32_t* tiles = p.item_tiles + item * p.n_kt;

  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sQ = sbase + kWarps * S::kWarpBytes;
  const uint32_t sW = sbase + warp * S::kWarpBytes;  // this warp's ring

  // ---- Q: 16 packed rows -> smem (zero for padding rows) ----
  for (int idx = tid; idx < kDecodeRows * S::kChunks; idx += kThreads) {
    int r = idx / S::kChunks, c = idx % S::kChunks;
    int P = geo.rt * kDecodeRows + r;
    int qi = P / p.G, h = geo.g * p.G + P % p.G;
    uint32_t dst = sQ + swz<D>(r, c);
    if (qi < geo.q_len) {
      int64_t qrow = p.cu_q ? (int64_t)p.cu_q[geo.b] + qi : (int64_t)qi;
      int64_t bo = p.cu_q ? 0 : (int64_t)geo.b;
      cp_async16(dst, p.q + bo * p.q_sb + qrow * p.q_ss + (int64_t)h * p.q_sh + c * 8);
    } else {
      asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0));
    }
  }
  cp_async_commit();
  if (KV2 && p.append && geo.rt == 0 && split == 0) append_active<D>(p, geo.b, geo.g, geo.lc, geo.q_len, tid, kThreads);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + S::kBarOff) + warp * kWarpStages;  // this warp's stages
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kBarOff + kWarps * kWarpStages * 8);
  if (TMA) {
    if (lane < kWarpStages) tc::mbar_init(kv_full + lane, 1);
    if (tid == 0) *abort_flag = 0;
    tc::fence_mbar_init();
    __syncwarp();
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmk);
      tc::tma_prefetch_desc(&tmv);
    }
  }
  uint32_t kv_phase = 0;  // TMA mode: parity of each stage's next completion

  // ---- this warp's chunks: c = warp, warp + 4, ... of the split ----
  const int n_chunks = (t_end - t_begin) * (kKeysPerTile / kChunkKeys);
  const int my_chunks = n_chunks > warp ? (n_chunks - warp + kWarps - 1) / kWarps : 0;
  const bool paged_fast = p.block_table && (p.page_size % kChunkKeys) == 0;
  // Chunk descriptors (first key, partial flag, page) are computed by the lane
  // whose index matches the chunk's position in a batch of 32, half a batch
  // ahead, and fetched with a shuffle: no global-memory load sits between a
  // chunk's turn and its copies.
  auto chunk_desc = [&](int k, int& kj0_, int& pg_) {
    kj0_ = -1;
    pg_ = 0;
    if (k >= my_chunks) return;
    const int c = warp + k * kWarps;
    const int e = __ldg(tiles + t_begin + c / (kKeysPerTile / kChunkKeys));
    kj0_ = ((e >> 1) * kKeysPerTile + (c % (kKeysPerTile / kChunkKeys)) * kChunkKeys) * 2 + (e & 1);
    const int kj = (e >> 1) * kKeysPerTile + (c % (kKeysPerTile / kChunkKeys)) * kChunkKeys;
    if (paged_fast && kj < geo.lc) pg_ = __ldg(p.block_table + (int64_t)geo.b * p.bt_stride + kj / p.page_size);
  };
  int dk_cur, dp_cur, dk_next, dp_next;  // this lane's descriptor in the current / next batch
  chunk_desc(lane, dk_cur, dp_cur);
  chunk_desc(32 + lane, dk_next, dp_next);
  auto chunk_key0 = [&](int k, bool& partial, bool& live, int& pg) -> int {
    const int src = k & 31;
    const bool cur = ((k >> 5) & 1) == 0;  // batches alternate between the two register sets
    const int code = __shfl_sync(0xffffffffu, cur ? dk_cur : dk_next, src);
    pg = __shfl_sync(0xffffffffu, cur ? dp_cur : dp_next, src);
    partial = (code & 1) != 0;
    const int kj0 = code >> 1;
    live = (kj0 <= geo.jhi) && (kj0 + kChunkKeys - 1 >= geo.jlo) && (kj0 < geo.kv_len);
    return kj0;
  };
  // lane l copies 16-byte chunk (l % 16) of rows 2i + l / 16 (i = 0..7) of K and V:
  // each instruction covers two whole rows (D = 128) or four (D = 64)
  auto load_chunk = [&](int k) {
    bool partial, live;
    int pg;
    const int kj0 = chunk_key0(k, partial, live, pg);
    if (!live) return;
    if (TMA && KV2 && kj0 >= geo.lc) return;  // active rows only: filled by the warp
    if (TMA) {
      if (lane == 0) {
        const int st = k % kWarpStages;
        int row, outer;
        if (p.block_table) {
          if ((unsigned)pg >= (unsigned)p.num_pages) {
            record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)pg);
            pg = 0;
          }
          row = kj0 % p.page_size;
          outer = pg;
        } else {
          row = (p.cu_k ? p.cu_k[geo.b] : 0) + kj0;
          outer = p.cu_k ? 0 : geo.b;
        }
        unsigned char* dst = smem + warp * S::kWarpBytes + st * S::kStageBytes;
        // this warp's reads of the stage (previous chunk) precede the copy
        tc::fence_proxy_async_smem();
        tc::mbar_arrive_expect_tx(kv_full + st, S::kStageBytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tc::tma_load_4d(dst + hf * (kChunkKeys * 128), &tmk, kv_full + st, hf * 64, geo.g, row, outer);
          tc::tma_load_4d(dst + S::kKvBytes + hf * (kChunkKeys * 128), &tmv, kv_full + st, hf * 64, geo.g, row,
                          outer);
        }
      }
      return;
    }
    const uint32_t sK = sW + (k % kWarpStages) * S::kStageBytes;
    const uint32_t sV = sK + S::kKvBytes;
    constexpr int kRowsPerInstr = 32 / S::kChunks;
    const int c = lane % S::kChunks, r0 = lane / S::kChunks;
    const uint16_t* kbase = nullptr;
    const uint16_t* vbase = nullptr;
    if (paged_fast) {
      if ((unsigned)pg >= (unsigned)p.num_pages) {
        record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)pg);
        pg = 0;
      }
      const int64_t row0 = kj0 % p.page_size;
      kbase = p.k + (int64_t)pg * p.k_sb + row0 * p.k_ss + (int64_t)geo.g * p.k_sh;
      vbase = p.v + (int64_t)pg * p.v_sb + row0 * p.v_ss + (int64_t)geo.g * p.v_sh;
    }
#pragma unroll
    for (int i = 0; i < kChunkKeys / kRowsPerInstr; ++i) {
      const int r = i * kRowsPerInstr + r0;
      const int j = min(kj0 + r, geo.kv_len - 1);
      const uint16_t* kr;
      const uint16_t* vr;
      if (paged_fast && kj0 + r < geo.lc) {
        kr = kbase + (int64_t)r * p.k_ss;
        vr = vbase + (int64_t)r * p.v_ss;
      } else {
        if constexpr (KV2) {
          kr = kv_src_row(p, false, geo.b, geo.g, j, geo.lc);
          vr = kv_src_row(p, true, geo.b, geo.g, j, geo.lc);
        } else {
          kr = kv_row(p, p.k, p.k_sb, p.k_ss, p.k_sh, geo.b, geo.g, j);
          vr = kv_row(p, p.v, p.v_sb, p.v_ss, p.v_sh, geo.b, geo.g, j);
        }
      }
      cp_async16(sK + swz<D>(r, c), kr + c * 8);
      cp_async16(sV + swz<D>(r, c), vr + c * 8);
    }
  };

  // TMA mode, two-source form: rows [r0, 16) of a chunk that holds active
  // rows are written by the warp itself when its turn comes: active rows from
  // k_new / v_new, rows past the keys as zeros (r0 = 0 for a chunk of active
  // rows only; for a chunk that starts in the cache the TMA copy brought the
  // cached rows, and r0 is the first active row).
  auto fill_chunk = [&](int k, int kj0, int r0) {
    const uint32_t sK = sW + (k % kWarpStages) * S::kStageBytes;
    for (int idx = lane + r0 * S::kChunks; idx < kChunkKeys * S::kChunks; idx += 32) {
      const int r = idx / S::kChunks, c = idx % S::kChunks;
      const int j = kj0 + r;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (j < geo.kv_len) {
        kv = __ldg(reinterpret_cast<const uint4*>(kv_src_row(p, false, geo.b, geo.g, j, geo.lc) + c * 8));
        vv = __ldg(reinterpret_cast<const uint4*>(kv_src_row(p, true, geo.b, geo.g, j, geo.lc) + c * 8));
      }
      const uint32_t o = swz_tma(r, c);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(sK + o), "r"(kv.x), "r"(kv.y), "r"(kv.z),
                   "r"(kv.w));
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(sK + S::kKvBytes + o), "r"(vv.x), "r"(vv.y),
                   "r"(vv.z), "r"(vv.w));
    }
    __syncwarp();
  };

  // Fragment roles: keys (and head-dim) on the mma M side, the 8 packed
  // query rows on N.  Lane = 4 g + c holds S^T[key g, g+8][row 2c, 2c+1] and
  // O^T[d 16m + g, + 8][row 2c, 2c+1].
  const int g8 = lane >> 2, c4 = lane & 3;
  int qi_r[2], h_r[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    int P = geo.rt * kDecodeRows + 2 * c4 + e;
    qi_r[e] = P / p.G;
    h_r[e] = geo.g * p.G + P % p.G;
  }
  // the first chunks go out before Q is waited for, so their latency overlaps
#pragma unroll
  for (int k = 0; k < kWarpStages - 1; ++k) {
    if (k < my_chunks) load_chunk(k);
    if (!TMA) cp_async_commit();
  }
  if (TMA) cp_async_wait<0>();       // this thread's Q copies have landed
  else cp_async_wait<kWarpStages - 1>();
  __syncthreads();                   // ... and everyone else's
  // Q^T as the B operand: [16 d x 8 rows] per k-step, two k-steps per ldmatrix.x4
  uint32_t qb[D / 16][2];
#pragma unroll
  for (int ks = 0; ks < D / 16; ks += 2) {
    const int mi = lane >> 3;
    ldsm_x4(sQ + swz<D>(lane & 7, 2 * ks + mi), qb[ks][0], qb[ks][1], qb[ks + 1][0], qb[ks + 1][1]);
  }
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o_acc[D / 16][4];
#pragma unroll
  for (int n = 0; n < D / 16; ++n) o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;

  bool ok = true;
  for (int k = 0; k < my_chunks; ++k) {
    if (!TMA) cp_async_wait<kWarpStages - 2>();
    __syncwarp();
    if (k + kWarpStages - 1 < my_chunks) load_chunk(k + kWarpStages - 1);
    if (!TMA) cp_async_commit();
    // half a batch past a batch start, the batch after next replaces the one just finished
    if ((k & 31) == 16 && k >= 32) {
      if (((k >> 5) & 1) == 0) chunk_desc((k & ~31) + 32 + lane + 0, dk_next, dp_next);
      else chunk_desc((k & ~31) + 32 + lane, dk_cur, dp_cur);
    }
    bool partial, live;
    int pg_unused;
    const int kj0 = chunk_key0(k, partial, live, pg_unused);
    if (!live) continue;
    if (TMA) {
      const int st = k % kWarpStages;
      if (KV2 && kj0 >= geo.lc) {
        fill_chunk(k, kj0, 0);  // no copy was issued for this stage: its barrier phase is unchanged
      } else {
        if (!tc::mbar_wait(kv_full + st, (kv_phase >> st) & 1, abort_flag)) {
          ok = false;
          break;
        }
        kv_phase ^= 1u << st;
        if (KV2 && kj0 + kChunkKeys > geo.lc) {
          fill_chunk(k, kj0, geo.lc - kj0);  // the active rows over the copied cache rows
        } else if (kj0 + kChunkKeys > geo.kv_len) {
          // a sequence's last chunk: the box also brought the page's unused
          // rows, which may hold anything (and P = 0 times a NaN is a NaN):
          // zero those V rows
          zero_rows_from<D>(sW + st * S::kStageBytes + S::kKvBytes, geo.kv_len - kj0, lane);
        }
      }
    }
    const uint32_t sK = sW + (k % kWarpStages) * S::kStageBytes;
    const uint32_t sV = sK + S::kKvBytes;

    // ---- S^T = K Q^T : 16 keys x 8 rows, two accumulator chains ----
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int mi = lane >> 3;
      uint32_t a[4];
      const int kr = (lane & 7) + 8 * (mi & 1), kc = 2 * ks + (mi >> 1);
      ldsm_x4(sK + (TMA ? swz_tma(kr, kc) : swz<D>(kr, kc)), a[0], a[1], a[2], a[3]);
      if (ks & 1) mma_bf16<F16>(sb, a, qb[ks][0], qb[ks][1]);
      else mma_bf16<F16>(sa, a, qb[ks][0], qb[ks][1]);
    }
    float sc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] = sa[e] + sb[e];
    // ---- logit transform (log2 units); element e: key g8 + 8 (e >> 1), row 2 c4 + (e & 1) ----
    // FULL chunk without an additive term: only scale (and soft-cap) apply
    const bool plain = !partial && p.mask_kind == FA_MASK_NONE && !p.alibi;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = kj0 + g8 + 8 * (e >> 1);
      const int rr = e & 1;
      if (plain) {
        sc[e] = p.softcap > 0.f ? softcap_log2(sc[e] * p.scale, p.softcap, p.inv_softcap) : sc[e] * p.scale_log2;
      } else if (qi_r[rr] >= geo.q_len) {
        sc[e] = -INFINITY;  // padding row: never read the mask out of range
      } else {
        sc[e] = logit_log2(p, sc[e], geo.b, h_r[rr], qi_r[rr], j, geo.off, geo.kv_len);
      }
    }
    // ---- online softmax per row (a column of S^T), -inf guarded ----
    float alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float mx = fmaxf(sc[rr], sc[rr + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[rr], mx);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[rr] = fast_exp2(m_run[rr] - m_ref);
      m_run[rr] = m_new;
      sc[rr] = fast_exp2(sc[rr] - m_ref);
      sc[rr + 2] = fast_exp2(sc[rr + 2] - m_ref);
      l_run[rr] = l_run[rr] * alpha[rr] + sc[rr] + sc[rr + 2];
    }
#pragma unroll
    for (int n = 0; n < D / 16; ++n) {
      o_acc[n][0] *= alpha[0]; o_acc[n][1] *= alpha[1];
      o_acc[n][2] *= alpha[0]; o_acc[n][3] *= alpha[1];
    }
    // ---- P^T (C layout) -> B operand [16 keys x 8 rows] by an 8x8 transpose ----
    const uint32_t pb0 = movmatrix_t(pack_bf16<F16>(sc[0], sc[1]));  // keys 0..7
    const uint32_t pb1 = movmatrix_t(pack_bf16<F16>(sc[2], sc[3]));  // keys 8..15
    // ---- O^T += V^T P^T : per 16 head-dim values, one mma over the 16 keys ----
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int mi = lane >> 3;
      uint32_t a[4];
      const int vr = (lane & 7) + 8 * (mi >> 1), vc = 2 * mt + (mi & 1);
      ldsm_x4_t(sV + (TMA ? swz_tma(vr, vc) : swz<D>(vr, vc)), a[0], a[1], a[2], a[3]);
      mma_bf16<F16>(o_acc[mt], a, pb0, pb1);
    }
  }
  cp_async_wait<0>();
  if (TMA && !ok && !*abort_flag) {
    *abort_flag = 1;
    record_error(p, FA_ERR_DEVICE_TIMEOUT, 22);
  }
  __syncthreads();
  if (TMA && *abort_flag) {
    // copies may still be landing in this warp's ring: let them, then leave
    // without touching shared memory or results
    if (lane < kWarpStages) tc::mbar_wait_drain(kv_full + lane, (kv_phase >> lane) & 1, 100000000ull);
    return;
  }

  decode_finish<D, F16>(p, geo, item, split, single, smem, reinterpret_cast<float*>(smem + kWarps * S::kWarpBytes), tid,
                   m_run, l_run, o_acc);
}

// Merge the splits of items that had more than one: LSE = logsumexp of the
// split LSEs (all -inf -> -inf), O = sum_s exp(LSE_s - LSE) O_s (0 if empty).
template <int D, bool F16>
__global__ void __launch_bounds__(32 * kDecodeRows) combine_kernel(const Params p) {
  const int64_t item = blockIdx.x;
  const int count = p.item_count[item];
  if (count <= p.tiles_per_split) return;
  const int n_eff = (count + p.tiles_per_split - 1) / p.tiles_per_split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemGeo geo = item_geo(p, item);
  const int row = warp;  // one warp per packed row
  uint16_t* optr; float* lptr; bool valid;
  out_ptrs(p, geo, geo.rt * kDecodeRows + row, optr, lptr, valid);
  if (!valid) return;
  const int64_t base = item * p.n_splits * kDecodeRows + row;
  float M = -INFINITY;
  for (int s = 0; s < n_eff; ++s) M = fmaxf(M, p.part_lse[base + (int64_t)s * kDecodeRows]);
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_eff; ++s) {
      float ls = p.part_lse[base + (int64_t)s * kDecodeRows];
      float w = __expf(ls - M);
      L += w;
      const float* po = p.part_o + (base + (int64_t)s * kDecodeRows) * D + lane * kPer;
#pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] += w * po[c];
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int c = 0; c < kPer; c += 2)
    *reinterpret_cast<uint32_t*>(optr + lane * kPer + c) = pack_bf16<F16>(acc[c] * inv, acc[c + 1] * inv);
  if (lane == 0) *lptr = (L > 0.f) ? (M + __logf(L)) : -INFINITY;
}

// Tensor maps for the TMA decode path: 4-D {d, Hkv, rows, outer} with a
// 16-row box; rows/outer are (row in page, page) for a paged cache, (row,
// sequence) or (packed row, 1) otherwise.  False when the layout has none.
template <int D>
bool decode_maps(const Params& p, CUtensorMap* mk, CUtensorMap* mv) {
  int64_t rows, outer, k_so, v_so;
  if (p.block_table) {
    if (p.page_size % kChunkKeys != 0) return false;
    rows = p.page_size;
    outer = p.num_pages;
    k_so = p.k_sb;
    v_so = p.v_sb;
  } else {
    rows = p.cache_len ? p.cache_cap : (p.cu_k ? p.tot_k : p.Sk);
    outer = p.cu_k ? 1 : p.n_seq;
    k_so = (outer == 1 || p.k_sb == 0) ? p.k_ss : p.k_sb;
    v_so = (outer == 1 || p.v_sb == 0) ? p.v_ss : p.v_sb;
  }
  if (rows <= 0 || outer <= 0) return false;
  return encode_4d_bf16(mk, p.k, D, p.Hkv, rows, outer, p.k_sh, p.k_ss, k_so, 64, kChunkKeys,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, p.f16 != 0) &&
         encode_4d_bf16(mv, p.v, D, p.Hkv, rows, outer, p.v_sh, p.v_ss, v_so, 64, kChunkKeys,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, p.f16 != 0);
}

template <int D, bool F16, bool KV2>
cudaError_t launch_decode_v(const Params& p, cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_attn_end) {
  cudaError_t e;
  const int64_t grid = p.n_items * p.n_splits;
  using S = DecodeSmem<D>;
  CUtensorMap mk, mv;
  if (decode_maps<D>(p, &mk, &mv)) {
    e = ensure_smem_attr<decode_kernel<D, true, F16, KV2>>(S::kTotal);
    if (e != cudaSuccess) return e;
    if (ev_begin && (e = cudaEventRecord(ev_begin, st)) != cudaSuccess) return e;
    decode_kernel<D, true, F16, KV2><<<(unsigned)grid, kThreads, S::kTotal, st>>>(p, mk, mv);
  } else {
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
    e = ensure_smem_attr<decode_kernel<D, false, F16, KV2>>(S::kTotal);
    if (e != cudaSuccess) return e;
    if (ev_begin && (e = cudaEventRecord(ev_begin, st)) != cudaSuccess) return e;
    decode_kernel<D, false, F16, KV2><<<(unsigned)grid, kThreads, S::kTotal, st>>>(p, mk, mv);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess && ev_attn_end) e = cudaEventRecord(ev_attn_end, st);
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  combine_kernel<D, F16><<<(unsigned)p.n_items, 32 * kDecodeRows, 0, st>>>(p);
  return cudaGetLastError();
}

// KV2: keys from two sources (fa_fwd_kvcache), a separate instantiation so
// that the one-source kernels carry none of its code
template <int D, bool F16>
cudaError_t launch_decode_d(const Params& p, cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_attn_end) {
  return p.cache_len ? launch_decode_v<D, F16, true>(p, st, ev_begin, ev_attn_end)
                     : launch_decode_v<D, F16, false>(p, st, ev_begin, ev_attn_end);
}

}  // namespace

cudaError_t launch_decode(const Params& p, cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_attn_end) {
  if (p.n_items <= 0) {
    cudaError_t e = ev_begin ? cudaEventRecord(ev_begin, st) : cudaSuccess;
    return (e == cudaSuccess && ev_attn_end) ? cudaEventRecord(ev_attn_end, st) : e;
  }
  if (p.f16)
    return p.d == 64 ? launch_decode_d<64, true>(p, st, ev_begin, ev_attn_end)
                     : launch_decode_d<128, true>(p, st, ev_begin, ev_attn_end);
  return p.d == 64 ? launch_decode_d<64, false>(p, st, ev_begin, ev_attn_end)
                   : launch_decode_d<128, false>(p, st, ev_begin, ev_attn_end);
}

}  // namespace mfa
