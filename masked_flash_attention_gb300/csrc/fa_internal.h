// fa_internal.h -- parameters shared by the host planner and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace mfa {

constexpr int kKeysPerTile = 128;     // scheduler key tile
constexpr int kPrefillRows = 128;     // query rows per prefill item (tcgen05 M)
constexpr int kDecodeRows = 8;        // packed rows per decode item (mma N)
constexpr int kMaxTopkKeys = 16384;   // top-k preparation keeps all keys of a row in smem

// Division by a divisor fixed for a launch, as a multiply-high and a shift
// (T. Granlund and P. Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, with a rounded-up multiplier): exact for
// 0 <= n < 2^31.  Built on the host, applied on the device.
struct FastDiv {
  uint32_t d, mul, shr;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 0u, 0u};
  if (d > 1) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;  // ceil(log2 d)
    const uint64_t p = 31 + l;
    f.mul = (uint32_t)(((1ull << p) + d - 1) / d);
    f.shr = (uint32_t)(p - 32);
  }
  return f;
}

// Workspace header (first 256 bytes of the workspace).
struct WsHeader {
  uint32_t error;       // fa_status of the first device fault, 0 = none
  uint32_t error_info;  // detail of that fault
  uint32_t pad[2];
};
// The workspace's first kWsHeadBytes bytes are zero-filled by the caller
// before its first use: the header, then the prefill tail-split arrival
// counts (Params::tail_flags), which every launch leaves at zero again.
constexpr size_t kWsHeadBytes = 256;
constexpr size_t kTailFlagsOff = sizeof(WsHeader);

// mask summary byte values
enum : uint8_t { kMaskEmpty = 0, kMaskZero = 1, kMaskMixed = 2 };

// Everything the kernels need; passed by value (fits the 32 KB param space).
struct Params {
  // tensors (element strides; head-dim stride is 1)
  const uint16_t* q; const uint16_t* k; const uint16_t* v;
  uint16_t* o; float* lse;
  int64_t q_sb, q_ss, q_sh;
  int64_t k_sb, k_ss, k_sh;  // paged: k_sb = page stride, k_ss = row-in-page stride
  int64_t v_sb, v_ss, v_sh;
  int64_t o_sb, o_ss, o_sh;
  int64_t lse_sb, lse_sh, lse_ss;
  const int32_t* cu_q;   // nullable
  const int32_t* cu_k;   // nullable
  const int32_t* block_table;  // nullable
  int64_t bt_stride;
  int32_t page_size, num_pages;

  int32_t n_seq, Sq, Sk;  // Sq/Sk: fixed lengths, or max lengths for varlen
  int64_t tot_q, tot_k;   // rows of packed Q / K (varlen), for device-side checks
  int32_t Hq, Hkv, G, d;
  int32_t f16;        // q, k, v, out are fp16 (else bf16)
  float scale;        // natural-log units
  float scale_log2;   // scale * log2(e)
  float softcap;      // 0 = off
  float inv_softcap;  // 1 / softcap (0 when off)
  const float* alibi; // [Hq] ALiBi slopes (natural-log units), null = off
  int32_t causal, wl, wr;

  // two key sources (fa_fwd_kvcache): sequence b's keys are cache rows
  // [0, cache_len[b]) (k / v) followed by its active rows in k_new / v_new,
  // laid out like q; null cache_len = one source
  const int32_t* cache_len;
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t kn_sb, kn_ss, kn_sh, vn_sb, vn_ss, vn_sh;
  int32_t cache_cap;  // cache rows a sequence may hold (block table width x page, or padded length)
  int32_t append;     // write the active rows into the cache

  // backward (fa_bwd): dO and Delta = rowsum(dO * O) (workspace, LSE layout);
  // dq like q, dk / dv like k / v
  const uint16_t* dout;
  int64_t do_sb, do_ss, do_sh;
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  int64_t dq_sb, dq_ss, dq_sh, dk_sb, dk_ss, dk_sh, dv_sb, dv_ss, dv_sh;
  float* delta;

  // additive mask
  int32_t mask_kind;
  const float* mask; int64_t m_sb, m_sh, m_sq, m_sk; int32_t m_nb, m_nh;
  const float* z; int64_t z_sb, z_sh, z_sk; int32_t keep_window;

  // scheduler
  int32_t path;
  // 1: the prefill kernel derives each unit's key tiles from the pair rules
  // (no dense or top-k mask), so no scheduler kernel runs and its lists are
  // not written; the kernel's first CTA writes the counters
  int32_t sched_inline;
  FastDiv div_units;  // prefill unit index -> row tile: n_seq * Hq
  FastDiv div_hq;     // -> sequence: Hq
  int32_t rows_per_tile, n_row_tiles, n_heads_sched, n_kt;
  int64_t n_items;
  int32_t* item_count;   // [n_items]
  int32_t* item_tiles;   // [n_items][n_kt]
  unsigned long long* stats;  // [3]
  uint8_t* mask_summary; // [m_nb][m_nh][n_row_tiles][n_kt]
  int32_t* topk_e;       // [n_seq][Hq][Sk]: first query row at which key j is dropped
  int32_t* topk_tile_maxe;  // [n_seq][Hq][n_kt] (few-row path)
  uint64_t* topk_runs;   // [n_seq][Hq][runs][2048]: sorted runs of (z order << 32 | index) words
  int32_t* topk_rank;    // [n_seq][Hq][Sk]: key of rank t (0 = best)
  int32_t* topk_rho;     // [n_seq][Hq][Sk]: rank of key j
  uint2* topk_list;      // [n_items][n_kt * 128]: gathered keys of each unit (many-row path)
  int32_t* topk_full;    // [n_items]: leading gathered tiles whose keys every row of the unit keeps

  // prefill grid and its tail split: the persistent grid takes the units in
  // rounds of prefill_grid; when the last round holds tail_units units (and
  // at most half the grid), each of them is cut into two pieces over the two
  // halves of its key tiles, run by two CTAs of that round; each piece
  // stores its normalised O and log2-sum-exp (tail_part: per piece, O as
  // [d][128 rows] then [2 warpgroups][128 rows], fp32), and the piece that
  // finishes second merges the two and writes the output.  tail_flags: one
  // 2-bit arrival count per (tail unit, softmax warpgroup), in the
  // workspace's zero-filled head, returned to zero by the merging piece.
  int32_t prefill_grid, tail_round, tail_units;
  float* tail_part;
  uint32_t* tail_flags;

  // decode split-KV
  int32_t n_splits, tiles_per_split;
  float* part_o;    // [n_items][n_splits][16][d]
  float* part_lse;  // [n_items][n_splits][16]

  WsHeader* ws;
  uint32_t debug_flags;

  // debug dump (fa_fwd_debug_dump): for the unit (dump_b, dump_h, dump_rt)
  // the prefill kernel's debug instantiation writes, per entry it of the
  // unit's key-tile list, raw S [it][row][key] and P [n_kt + it][row][key]
  // (fp32; P as rounded for PV) and the exponent reference of each row
  // [2 n_kt x 128 x 128 + it x 128 + row], and the unit's list into the
  // work list; null = off
  float* dump;
  int32_t dump_b, dump_h, dump_rt;
};

// ---- launchers (defined in the .cu files; all enqueue on `st`) ----
cudaError_t launch_mask_summary(const Params& p, cudaStream_t st);
// Top-k preparation (topk.cu): expiry rows, then the gathered key lists and
// counts (many-row path) or the per-tile maxima (few-row path).
cudaError_t launch_topk_prep(const Params& p, cudaStream_t st);
int topk_n_runs(int Sk);
// NVTX ranges around the forward and backward stages (on unless a caller on
// this thread turns them off; fa_fwd_noalloc does, around its call).
extern thread_local bool g_trace_ranges;
cudaError_t launch_classify(const Params& p, cudaStream_t st);
// The attention launchers record `ev_begin` (if not null) on the stream right
// before the kernel itself is enqueued, after all host-side preparation.
cudaError_t launch_decode(const Params& p, cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_attn_end);
cudaError_t launch_prefill(const Params& p, cudaStream_t st, cudaEvent_t ev_begin);
// Host: the prefill kernel's persistent grid for this device and the split of
// its last round (Params::prefill_grid, tail_round, tail_units).
void plan_prefill_grid(Params& p);
cudaError_t launch_prefill_f16(const Params& p, cudaStream_t st, cudaEvent_t ev_begin);  // p.f16 inputs
cudaError_t launch_backward(const Params& p, cudaStream_t st, cudaEvent_t ev_begin);
// dK/dV and dQ of the backward on tcgen05; *launched = false (nothing
// enqueued) when a tensor map cannot describe the layout
cudaError_t launch_bwd_tc(const Params& p, cudaStream_t st, bool* launched);

}  // namespace mfa
