// api.cu -- the C ABI: argument validation, planning, workspace layout and
// kernel launches.  Argument rules follow the vLLM pull request 11277
// flash_attn_varlen_func argument list (q, k, v, out, cu_seqlens_q/k,
// max_seqlen_q/k, softmax scale, causal, window, block_table, softcap) and
// InfiniTrain pull request 193 ("Framework 与 autograd": MHA when Hq == Hkv,
// GQA/MQA when Hq % Hkv == 0, an error otherwise; review comments: an
// unsupported feature must report an error, and a wrong dtype must be caught
// at the entry).  No path here falls back to anything: an argument the kernels
// cannot take is an error code.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "fa_internal.h"

using namespace mfa;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// An activation/cache tensor: bf16 or fp16, rank, unit head-dim stride,
// other strides multiples of 8 elements (16 bytes), 16-byte aligned base.
int check_bf16(const fa_tensor* t, int ndim) {
  if (!t || !t->data) return FA_ERR_INVALID_ARG;
  if ((t->dtype != FA_DTYPE_BF16 && t->dtype != FA_DTYPE_F16) || t->ndim != ndim) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return FA_ERR_INVALID_ARG;
  if (t->stride[ndim - 1] != 1) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < ndim - 1; ++i)
    if (t->stride[i] < 0 || (t->stride[i] % 8) != 0) return FA_ERR_INVALID_ARG;
  if (!aligned16(t->data)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int check_i32_vec(const fa_tensor* t, int64_t len) {
  if (!t || !t->data || t->dtype != FA_DTYPE_I32 || t->ndim != 1) return FA_ERR_INVALID_ARG;
  if (t->shape[0] != len || t->stride[0] != 1) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// The second key source of fa_fwd_kvcache (null for fa_fwd).
struct KvNew {
  const fa_tensor* k_new;
  const fa_tensor* v_new;
  const fa_tensor* cache_seqlens;
  int32_t append;
};

struct Plan {
  fa_plan pub;
  Params prm;
  size_t off_summary, off_topk_e, off_topk_maxe, off_topk_runs, off_topk_rank, off_topk_rho, off_topk_list,
      off_topk_full, off_part_o, off_part_lse, off_tail;
};

int make_plan(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
              const fa_tensor* lse, const fa_tensor* cu_q, const fa_tensor* cu_k,
              const fa_tensor* block_table, const fa_mask* mask, int32_t wl, int32_t wr,
              float softcap, float scale, int32_t causal, const fa_opts* opts, Plan* pl,
              const KvNew* kn = nullptr) {
  if (!q || !k || !v || !out || !lse || !opts || !pl) return FA_ERR_INVALID_ARG;
  memset(pl, 0, sizeof(*pl));
  Params& P = pl->prm;
  fa_plan& pub = pl->pub;
  const bool varlen_q = cu_q != nullptr;
  const bool varlen_k = cu_k != nullptr;
  const bool paged = block_table != nullptr;
  // page tables need per-sequence key counts: cu_seqlens_k, or the cached
  // counts of the two-source form (which takes no cu_seqlens_k)
  if (kn ? varlen_k : (paged && !varlen_k)) return FA_ERR_INVALID_ARG;
  int rc;

  // ---- Q ----
  int64_t n_seq, Sq, Hq, d;
  if (varlen_q) {
    if ((rc = check_bf16(q, 3))) return rc;
    if (!cu_q->data || cu_q->ndim != 1 || cu_q->shape[0] < 1) return FA_ERR_INVALID_ARG;
    n_seq = cu_q->shape[0] - 1;
    if ((rc = check_i32_vec(cu_q, n_seq + 1))) return rc;
    Sq = opts->max_seqlen_q;
    if (Sq < 0 || (Sq == 0 && q->shape[0] > 0)) return FA_ERR_INVALID_ARG;
    Hq = q->shape[1];
    d = q->shape[2];
    P.q_sb = 0; P.q_ss = q->stride[0]; P.q_sh = q->stride[1];
  } else {
    if ((rc = check_bf16(q, 4))) return rc;
    n_seq = q->shape[0];
    Sq = q->shape[1];
    Hq = q->shape[2];
    d = q->shape[3];
    P.q_sb = q->stride[0]; P.q_ss = q->stride[1]; P.q_sh = q->stride[2];
  }
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (Hq < 1) return FA_ERR_INVALID_ARG;

  // ---- K / V ----
  int64_t Sk, Hkv, page_size = 0, num_pages = 0;
  if (paged) {
    if ((rc = check_bf16(k, 4)) || (rc = check_bf16(v, 4))) return rc;
    num_pages = k->shape[0];
    page_size = k->shape[1];
    Hkv = k->shape[2];
    if (k->shape[3] != d || page_size < 1) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (v->shape[i] != k->shape[i]) return FA_ERR_INVALID_ARG;
    P.k_sb = k->stride[0]; P.k_ss = k->stride[1]; P.k_sh = k->stride[2];
    P.v_sb = v->stride[0]; P.v_ss = v->stride[1]; P.v_sh = v->stride[2];
    if (!block_table->data || block_table->dtype != FA_DTYPE_I32 || block_table->ndim != 2 ||
        block_table->shape[0] != n_seq || block_table->stride[1] != 1 || block_table->shape[1] < 1)
      return FA_ERR_INVALID_ARG;
    Sk = opts->max_seqlen_k;
    if (Sk < 0 || (!kn && Sk > block_table->shape[1] * page_size)) return FA_ERR_INVALID_ARG;
  } else if (varlen_k) {
    if ((rc = check_bf16(k, 3)) || (rc = check_bf16(v, 3))) return rc;
    Hkv = k->shape[1];
    if (k->shape[2] != d) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
      if (v->shape[i] != k->shape[i]) return FA_ERR_INVALID_ARG;
    P.k_sb = 0; P.k_ss = k->stride[0]; P.k_sh = k->stride[1];
    P.v_sb = 0; P.v_ss = v->stride[0]; P.v_sh = v->stride[1];
    Sk = opts->max_seqlen_k;
    if (Sk < 0 || (Sk == 0 && k->shape[0] > 0)) return FA_ERR_INVALID_ARG;
  } else {
    if ((rc = check_bf16(k, 4)) || (rc = check_bf16(v, 4))) return rc;
    if (k->shape[0] != n_seq) return FA_ERR_INVALID_ARG;
    Sk = k->shape[1];
    Hkv = k->shape[2];
    if (k->shape[3] != d) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (v->shape[i] != k->shape[i]) return FA_ERR_INVALID_ARG;
    P.k_sb = k->stride[0]; P.k_ss = k->stride[1]; P.k_sh = k->stride[2];
    P.v_sb = v->stride[0]; P.v_ss = v->stride[1]; P.v_sh = v->stride[2];
  }
  if (varlen_k && (rc = check_i32_vec(cu_k, n_seq + 1))) return rc;
  int64_t cache_cap = 0;
  if (kn) {
    // cache capacity per sequence; keys = cached + active, at most max_seqlen_k
    cache_cap = paged ? block_table->shape[1] * page_size : Sk;
    Sk = opts->max_seqlen_k;
    if (Sk < 0 || (Sk == 0 && Sq > 0 && n_seq > 0)) return FA_ERR_INVALID_ARG;
    if (!kn->k_new || !kn->v_new) return FA_ERR_INVALID_ARG;
    const fa_tensor* kv2[2] = {kn->k_new, kn->v_new};
    for (const fa_tensor* t : kv2) {
      if ((rc = check_bf16(t, (int)q->ndim))) return rc;
      if (t->dtype != q->dtype) return FA_ERR_INVALID_ARG;
      for (int i = 0; i < q->ndim; ++i) {
        const int64_t want = (i == q->ndim - 2) ? Hkv : q->shape[i];
        if (t->shape[i] != want) return FA_ERR_INVALID_ARG;
      }
    }
    if ((rc = check_i32_vec(kn->cache_seqlens, n_seq))) return rc;
    const fa_tensor *kt = kn->k_new, *vt = kn->v_new;
    if (varlen_q) {
      P.kn_sb = 0; P.kn_ss = kt->stride[0]; P.kn_sh = kt->stride[1];
      P.vn_sb = 0; P.vn_ss = vt->stride[0]; P.vn_sh = vt->stride[1];
    } else {
      P.kn_sb = kt->stride[0]; P.kn_ss = kt->stride[1]; P.kn_sh = kt->stride[2];
      P.vn_sb = vt->stride[0]; P.vn_ss = vt->stride[1]; P.vn_sh = vt->stride[2];
    }
    P.k_new = static_cast<const uint16_t*>(kt->data);
    P.v_new = static_cast<const uint16_t*>(vt->data);
    P.cache_len = static_cast<const int32_t*>(kn->cache_seqlens->data);
    P.cache_cap = (int32_t)(cache_cap < INT32_MAX ? cache_cap : INT32_MAX);
    P.append = kn->append ? 1 : 0;
  }
  // grouped-query heads: Hq a multiple of Hkv, otherwise an error
  if (Hkv < 1 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (Sq > INT32_MAX / 64 || Sk > INT32_MAX / 64 || n_seq > INT32_MAX / 64) return FA_ERR_INVALID_ARG;

  // ---- out / lse ----
  // one element type for q, k, v and out
  if (k->dtype != q->dtype || v->dtype != q->dtype || out->dtype != q->dtype) return FA_ERR_INVALID_ARG;
  if (out->ndim != q->ndim || !out->data) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < q->ndim; ++i)
    if (out->shape[i] != q->shape[i]) return FA_ERR_INVALID_ARG;
  if ((rc = check_bf16(out, out->ndim))) return rc;
  if (!lse->data || lse->dtype != FA_DTYPE_F32) return FA_ERR_INVALID_ARG;
  if (varlen_q) {
    if (lse->ndim != 2 || lse->shape[0] != Hq || lse->shape[1] != q->shape[0]) return FA_ERR_INVALID_ARG;
    P.lse_sb = 0; P.lse_sh = lse->stride[0]; P.lse_ss = lse->stride[1];
    P.o_sb = 0; P.o_ss = out->stride[0]; P.o_sh = out->stride[1];
  } else {
    if (lse->ndim != 3 || lse->shape[0] != n_seq || lse->shape[1] != Hq || lse->shape[2] != Sq)
      return FA_ERR_INVALID_ARG;
    P.lse_sb = lse->stride[0]; P.lse_sh = lse->stride[1]; P.lse_ss = lse->stride[2];
    P.o_sb = out->stride[0]; P.o_ss = out->stride[1]; P.o_sh = out->stride[2];
  }
  if ((reinterpret_cast<uintptr_t>(lse->data) & 3u) != 0) return FA_ERR_INVALID_ARG;

  // ---- scalars ----
  if (wl < -1 || wr < -1) return FA_ERR_INVALID_ARG;
  if (!(softcap >= 0.f) || !std::isfinite(softcap)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (scale <= 0.f) scale = 1.0f / std::sqrt((float)d);

  // ---- mask ----
  int mask_kind = mask ? mask->kind : FA_MASK_NONE;
  if (kn && mask_kind != FA_MASK_NONE) return FA_ERR_UNSUPPORTED;
  P.m_nb = P.m_nh = 1;
  if (mask_kind == FA_MASK_DENSE) {
    const fa_tensor& t = mask->t;
    if (!t.data || t.dtype != FA_DTYPE_F32) return FA_ERR_INVALID_ARG;
    if (varlen_q || varlen_k || paged) return FA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(t.data) & 3u) != 0) return FA_ERR_INVALID_ARG;
    if (t.ndim == 2) {
      if (t.shape[0] != Sq || t.shape[1] != Sk) return FA_ERR_INVALID_ARG;
      P.m_sb = 0; P.m_sh = 0; P.m_sq = t.stride[0]; P.m_sk = t.stride[1];
    } else if (t.ndim == 4) {
      if ((t.shape[0] != n_seq && t.shape[0] != 1) || (t.shape[1] != Hq && t.shape[1] != 1) ||
          t.shape[2] != Sq || t.shape[3] != Sk)
        return FA_ERR_INVALID_ARG;
      P.m_sb = t.stride[0]; P.m_sh = t.stride[1]; P.m_sq = t.stride[2]; P.m_sk = t.stride[3];
      P.m_nb = (t.shape[0] > 1 && t.stride[0] != 0) ? (int)n_seq : 1;
      P.m_nh = (t.shape[1] > 1 && t.stride[1] != 0) ? (int)Hq : 1;
    } else {
      return FA_ERR_INVALID_ARG;
    }
    P.mask = static_cast<const float*>(t.data);
  } else if (mask_kind == FA_MASK_TOPK) {
    const fa_tensor& t = mask->t;
    if (!t.data || t.dtype != FA_DTYPE_F32 || t.ndim != 3) return FA_ERR_INVALID_ARG;
    if (mask->keep_window < 1) return FA_ERR_INVALID_ARG;
    if (varlen_q || varlen_k || paged) return FA_ERR_UNSUPPORTED;
    if (wl >= 0 || wr >= 0) return FA_ERR_UNSUPPORTED;
    if (Sk > kMaxTopkKeys) return FA_ERR_UNSUPPORTED;
    if (t.shape[0] != n_seq || t.shape[1] != Hq || t.shape[2] != Sk) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(t.data) & 3u) != 0) return FA_ERR_INVALID_ARG;
    P.z = static_cast<const float*>(t.data);
    P.z_sb = t.stride[0]; P.z_sh = t.stride[1]; P.z_sk = t.stride[2];
    P.keep_window = mask->keep_window;
  } else if (mask_kind != FA_MASK_NONE) {
    return FA_ERR_INVALID_ARG;
  }

  // ---- fill the scalar part of Params ----
  P.q = static_cast<const uint16_t*>(q->data);
  P.k = static_cast<const uint16_t*>(k->data);
  P.v = static_cast<const uint16_t*>(v->data);
  P.o = static_cast<uint16_t*>(out->data);
  P.lse = static_cast<float*>(lse->data);
  P.cu_q = varlen_q ? static_cast<const int32_t*>(cu_q->data) : nullptr;
  P.cu_k = varlen_k ? static_cast<const int32_t*>(cu_k->data) : nullptr;
  P.block_table = paged ? static_cast<const int32_t*>(block_table->data) : nullptr;
  P.bt_stride = paged ? block_table->stride[0] : 0;
  P.page_size = (int32_t)page_size;
  P.num_pages = (int32_t)num_pages;
  P.tot_q = varlen_q ? q->shape[0] : 0;
  P.tot_k = (varlen_k && !paged) ? k->shape[0] : 0;
  P.n_seq = (int32_t)n_seq;
  P.Sq = (int32_t)Sq;
  P.Sk = (int32_t)Sk;
  P.Hq = (int32_t)Hq;
  P.Hkv = (int32_t)Hkv;
  P.G = (int32_t)(Hq / Hkv);
  P.d = (int32_t)d;
  P.scale = scale;
  P.scale_log2 = scale * 1.4426950408889634f;
  P.softcap = softcap;
  P.inv_softcap = softcap > 0.f ? 1.f / softcap : 0.f;
  P.causal = causal ? 1 : 0;
  P.f16 = q->dtype == FA_DTYPE_F16 ? 1 : 0;
  P.wl = wl;
  P.wr = wr;
  P.mask_kind = mask_kind;
  P.debug_flags = opts->debug_flags;
  P.alibi = static_cast<const float*>(opts->alibi_slopes);

  // ---- path and tile geometry ----
  // Few query rows per K/V head (decode): the 16-row split-KV kernel.  Many
  // rows: the tcgen05 kernel, which reads Q/K/V through TMA tensor maps and so
  // needs non-zero strides on every dimension of extent > 1 and a contiguous
  // (non-paged) K/V.
  const int G = P.G;
  bool tma_ok = !paged;
  if (!varlen_q && n_seq > 1 && P.q_sb == 0) tma_ok = false;
  if (!varlen_k && !paged && n_seq > 1 && (P.k_sb == 0 || P.v_sb == 0)) tma_ok = false;
  if ((Hq > 1 && P.q_sh == 0) || (Hkv > 1 && (P.k_sh == 0 || P.v_sh == 0))) tma_ok = false;
  if (P.q_ss == 0 || P.k_ss == 0 || P.v_ss == 0) tma_ok = false;
  const bool prefill = tma_ok && !kn && Sq * (int64_t)G > 64;  // two sources: decode kernel
  if (prefill) {
    P.path = FA_PATH_PREFILL;
    P.rows_per_tile = kPrefillRows;
    P.n_heads_sched = (int32_t)Hq;
    P.n_row_tiles = ceil_div(Sq, kPrefillRows);
  } else {
    P.path = FA_PATH_DECODE;
    P.rows_per_tile = kDecodeRows;
    P.n_heads_sched = (int32_t)Hkv;
    P.n_row_tiles = ceil_div(Sq * G, kDecodeRows);
  }
  // the top-k prefill gathers K/V rows through a 2-D view [B * Sk rows, one
  // row of all K/V heads]: each batch's rows must follow the previous batch's
  // rows and a row's heads must fit inside the row stride
  if (P.path == FA_PATH_PREFILL && mask_kind == FA_MASK_TOPK) {
    const bool kv_rows = (n_seq == 1 || (P.k_sb == Sk * P.k_ss && P.v_sb == Sk * P.v_ss)) &&
                         (Hkv - 1) * P.k_sh + d <= P.k_ss && (Hkv - 1) * P.v_sh + d <= P.v_ss;
    if (!kv_rows) return FA_ERR_UNSUPPORTED;
  }
  // prefill carries ALiBi without a mask or with a dense one, not with top-k
  // (decode: any)
  if (P.path == FA_PATH_PREFILL && P.alibi && mask_kind == FA_MASK_TOPK) return FA_ERR_UNSUPPORTED;
  // without a dense or top-k mask the pair rules alone decide every tile: the
  // prefill kernel classifies its units' tiles itself and no scheduler kernel runs
  P.sched_inline = (P.path == FA_PATH_PREFILL && mask_kind == FA_MASK_NONE) ? 1 : 0;
  P.n_kt = ceil_div(Sk, kKeysPerTile);
  P.n_items = n_seq * (int64_t)P.n_heads_sched * P.n_row_tiles;
  P.div_units = make_fastdiv((uint32_t)(n_seq * Hq > 0 ? n_seq * Hq : 1));
  P.div_hq = make_fastdiv((uint32_t)(Hq > 0 ? Hq : 1));
  if (Sq == 0 || n_seq == 0) P.n_items = 0;

  // split-KV factor: enough CTAs to cover the GPU a few times over
  int n_kt_alloc = P.n_kt > 0 ? P.n_kt : 1;
  P.n_splits = 1;
  P.tiles_per_split = n_kt_alloc;
  if (P.path == FA_PATH_DECODE && P.n_items > 0 && n_kt_alloc > 8) {
    // (at most 8 key tiles: one CTA per item, no combine pass -- splitting
    // such short rows costs more in launches than it saves)
    const int64_t target_ctas = 152 * 16;
    if (P.n_items < target_ctas / 2) {
      int64_t tps = (P.n_items * (int64_t)n_kt_alloc + target_ctas - 1) / target_ctas;
      tps = tps < 1 ? 1 : (tps > 8 ? 8 : tps);
      P.tiles_per_split = (int32_t)tps;
      P.n_splits = ceil_div(n_kt_alloc, tps);
    }
  }

  // ---- workspace layout ----
  size_t off = align_up(sizeof(WsHeader));
  pub.off_stats = off;
  off = align_up(off + 3 * sizeof(long long));
  pub.off_counts = off;
  off = align_up(off + (size_t)P.n_items * 4);
  pub.off_tiles = off;
  off = align_up(off + (size_t)P.n_items * n_kt_alloc * 4);
  pl->off_summary = off;
  if (mask_kind == FA_MASK_DENSE) off = align_up(off + (size_t)P.m_nb * P.m_nh * P.n_row_tiles * n_kt_alloc);
  pl->off_topk_e = off;
  if (mask_kind == FA_MASK_TOPK) off = align_up(off + (size_t)n_seq * Hq * Sk * 4);
  pl->off_topk_maxe = off;
  if (mask_kind == FA_MASK_TOPK) off = align_up(off + (size_t)n_seq * Hq * n_kt_alloc * 4);
  pl->off_topk_runs = off;
  if (mask_kind == FA_MASK_TOPK) off = align_up(off + (size_t)n_seq * Hq * topk_n_runs((int)Sk) * 2048 * 8);
  pl->off_topk_rank = off;
  if (mask_kind == FA_MASK_TOPK) off = align_up(off + (size_t)n_seq * Hq * Sk * 4);
  pl->off_topk_rho = off;
  if (mask_kind == FA_MASK_TOPK) off = align_up(off + (size_t)n_seq * Hq * Sk * 4);
  pl->off_topk_list = off;
  if (mask_kind == FA_MASK_TOPK && P.path == FA_PATH_PREFILL)
    off = align_up(off + (size_t)P.n_items * n_kt_alloc * kKeysPerTile * 8);
  pl->off_topk_full = off;
  if (mask_kind == FA_MASK_TOPK && P.path == FA_PATH_PREFILL) off = align_up(off + (size_t)P.n_items * 4);
  pl->off_part_o = off;
  if (P.n_splits > 1) off = align_up(off + (size_t)P.n_items * P.n_splits * kDecodeRows * d * 4);
  pl->off_part_lse = off;
  if (P.n_splits > 1) off = align_up(off + (size_t)P.n_items * P.n_splits * kDecodeRows * 4);
  // prefill: persistent grid and the split of its last round (mask-free units)
  P.prefill_grid = P.tail_round = P.tail_units = 0;
  if (P.path == FA_PATH_PREFILL && P.n_items > 0) plan_prefill_grid(P);
  pl->off_tail = off;
  if (P.tail_units > 0) off = align_up(off + (size_t)P.tail_units * 2 * (kPrefillRows * d + 256) * 4);

  pub.path = P.path;
  pub.n_seq = P.n_seq;
  pub.n_heads_sched = P.n_heads_sched;
  pub.n_row_tiles = P.n_row_tiles;
  pub.rows_per_tile = P.rows_per_tile;
  pub.keys_per_tile = kKeysPerTile;
  pub.n_k_tiles = n_kt_alloc;
  pub.n_splits = P.n_splits;
  pub.tiles_per_split = P.tiles_per_split;
  pub.tail_units = P.tail_units;
  pub.n_items = P.n_items;
  pub.off_topk_e = (mask_kind == FA_MASK_TOPK) ? pl->off_topk_e : 0;
  pub.off_topk_list = (mask_kind == FA_MASK_TOPK && P.path == FA_PATH_PREFILL) ? pl->off_topk_list : 0;
  // top-k: sort runs, ranks, expiry rows, then the gathered lists (prefill,
  // which replace the scheduler kernel) or the tile maxima (decode)
  pub.n_kernels = P.n_items == 0 ? 0
                  : P.sched_inline ? 1
                  : (mask_kind == FA_MASK_TOPK && P.path == FA_PATH_PREFILL) ? 5
                  : 2 + (P.n_splits > 1) + (mask_kind == FA_MASK_DENSE) + 4 * (mask_kind == FA_MASK_TOPK);
  pub.workspace_bytes = off;
  P.n_kt = n_kt_alloc;
  return FA_OK;
}

void bind_workspace(Plan* pl, void* ws) {
  unsigned char* base = static_cast<unsigned char*>(ws);
  Params& P = pl->prm;
  P.ws = reinterpret_cast<WsHeader*>(base);
  P.stats = reinterpret_cast<unsigned long long*>(base + pl->pub.off_stats);
  P.item_count = reinterpret_cast<int32_t*>(base + pl->pub.off_counts);
  P.item_tiles = reinterpret_cast<int32_t*>(base + pl->pub.off_tiles);
  P.mask_summary = base + pl->off_summary;
  P.topk_e = reinterpret_cast<int32_t*>(base + pl->off_topk_e);
  P.topk_tile_maxe = reinterpret_cast<int32_t*>(base + pl->off_topk_maxe);
  P.topk_runs = reinterpret_cast<uint64_t*>(base + pl->off_topk_runs);
  P.topk_rank = reinterpret_cast<int32_t*>(base + pl->off_topk_rank);
  P.topk_rho = reinterpret_cast<int32_t*>(base + pl->off_topk_rho);
  P.topk_list = reinterpret_cast<uint2*>(base + pl->off_topk_list);
  P.topk_full = reinterpret_cast<int32_t*>(base + pl->off_topk_full);
  P.part_o = reinterpret_cast<float*>(base + pl->off_part_o);
  P.part_lse = reinterpret_cast<float*>(base + pl->off_part_lse);
  P.tail_part = reinterpret_cast<float*>(base + pl->off_tail);
  P.tail_flags = reinterpret_cast<uint32_t*>(base + kTailFlagsOff);
}

// The device must be an sm_103 part (checked once per device).
int check_device() {
  static std::atomic<int> cached[64];  // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_NO_DEVICE;
  if (dev < 0 || dev >= 64) return FA_ERR_NO_DEVICE;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    c = (major == 10 && minor == 3) ? 1 : 2;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c == 1 ? FA_OK : FA_ERR_NO_DEVICE;
}


int run_plan(Plan& pl, const fa_opts* opts);  // enqueue a validated plan (below)

// fa_bwd: the forward's arguments (validated by make_plan, without mask or
// page table) plus dO, dq, dk, dv; Delta is appended to the workspace.
int make_plan_bwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                  const fa_tensor* lse, const fa_tensor* dout, const fa_tensor* dq, const fa_tensor* dk,
                  const fa_tensor* dv, const fa_tensor* cu_q, const fa_tensor* cu_k, int32_t wl, int32_t wr,
                  float softcap, float scale, int32_t causal, const fa_opts* opts, Plan* pl, size_t* off_delta) {
  int rc = make_plan(q, k, v, out, lse, cu_q, cu_k, nullptr, nullptr, wl, wr, softcap, scale, causal, opts, pl);
  if (rc != FA_OK) return rc;
  Params& P = pl->prm;
  const fa_tensor* qs[2] = {dout, dq};
  for (const fa_tensor* t : qs) {
    if ((rc = check_bf16(t, (int)q->ndim))) return rc;
    if (t->dtype != q->dtype) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < q->ndim; ++i)
      if (t->shape[i] != q->shape[i]) return FA_ERR_INVALID_ARG;
  }
  const fa_tensor* ks[2] = {dk, dv};
  for (const fa_tensor* t : ks) {
    if ((rc = check_bf16(t, (int)k->ndim))) return rc;
    if (t->dtype != q->dtype) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < k->ndim; ++i)
      if (t->shape[i] != k->shape[i]) return FA_ERR_INVALID_ARG;
  }
  auto strides = [](const fa_tensor* t, int64_t& sb, int64_t& ss, int64_t& sh) {
    if (t->ndim == 3) { sb = 0; ss = t->stride[0]; sh = t->stride[1]; }
    else { sb = t->stride[0]; ss = t->stride[1]; sh = t->stride[2]; }
  };
  strides(dout, P.do_sb, P.do_ss, P.do_sh);
  strides(dq, P.dq_sb, P.dq_ss, P.dq_sh);
  strides(dk, P.dk_sb, P.dk_ss, P.dk_sh);
  strides(dv, P.dv_sb, P.dv_ss, P.dv_sh);
  P.dout = static_cast<const uint16_t*>(dout->data);
  P.dq = static_cast<uint16_t*>(dq->data);
  P.dk = static_cast<uint16_t*>(dk->data);
  P.dv = static_cast<uint16_t*>(dv->data);
  const int64_t rows = cu_q ? q->shape[0] : (int64_t)P.n_seq * P.Sq;
  *off_delta = pl->pub.workspace_bytes;
  pl->pub.workspace_bytes = align_up(*off_delta + (size_t)rows * P.Hq * 4);
  pl->pub.n_kernels = (rows > 0 && P.Hq > 0) ? 3 : 0;
  return FA_OK;
}
}  // namespace

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported argument combination";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case FA_ERR_DEVICE_BOUNDS: return "device index out of range";
    case FA_ERR_DEVICE_VALUE: return "mask value not accepted (NaN, +inf, or a non-finite top-k score)";
    case FA_ERR_NO_DEVICE: return "no sm_103 device";
    default: return "unknown status";
  }
}

int fa_fwd_plan(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                const fa_tensor* lse, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                const fa_tensor* block_table, const fa_mask* mask, int32_t window_left,
                int32_t window_right, float softcap, float scale, int32_t causal,
                const fa_opts* opts, fa_plan* plan_out) {
  Plan pl;
  int rc = make_plan(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, window_left,
                     window_right, softcap, scale, causal, opts, &pl);
  if (rc == FA_OK && plan_out) *plan_out = pl.pub;
  return rc;
}

int fa_fwd_workspace_size(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                          const fa_tensor* out, const fa_tensor* lse, const fa_tensor* cu_seqlens_q,
                          const fa_tensor* cu_seqlens_k, const fa_tensor* block_table,
                          const fa_mask* mask, int32_t window_left, int32_t window_right,
                          float softcap, float scale, int32_t causal, const fa_opts* opts,
                          size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  Plan pl;
  int rc = make_plan(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, window_left,
                     window_right, softcap, scale, causal, opts, &pl);
  if (rc == FA_OK) *bytes = pl.pub.workspace_bytes;
  return rc;
}

int fa_fwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
           const fa_tensor* lse, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
           const fa_tensor* block_table, const fa_mask* mask, int32_t window_left,
           int32_t window_right, float softcap, float scale, int32_t causal, const fa_opts* opts) {
  Plan pl;
  int rc = make_plan(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table, mask, window_left,
                     window_right, softcap, scale, causal, opts, &pl);
  if (rc != FA_OK) return rc;
  return run_plan(pl, opts);
}

int fa_fwd_debug_dump(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                      const fa_tensor* lse, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                      int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
                      const fa_opts* opts, int32_t seq, int32_t head, int32_t row_tile, float* dump,
                      size_t dump_bytes) {
  Plan pl;
  int rc = make_plan(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, nullptr, nullptr, window_left, window_right,
                     softcap, scale, causal, opts, &pl);
  if (rc != FA_OK) return rc;
  Params& P = pl.prm;
  // the debug instantiations: prefill path, bf16, no ALiBi
  if (P.path != FA_PATH_PREFILL || P.f16 || P.alibi) return FA_ERR_UNSUPPORTED;
  if (!dump || seq < 0 || seq >= P.n_seq || head < 0 || head >= P.Hq || row_tile < 0 || row_tile >= P.n_row_tiles)
    return FA_ERR_INVALID_ARG;
  if (dump_bytes < fa_debug_dump_bytes(pl.pub.n_k_tiles)) return FA_ERR_INVALID_ARG;
  P.dump = dump;
  P.tail_units = 0;  // the debug instantiation runs every unit whole
  P.dump_b = seq;
  P.dump_h = head;
  P.dump_rt = row_tile;
  return run_plan(pl, opts);
}

size_t fa_debug_dump_bytes(int64_t n_k_tiles) {
  return n_k_tiles <= 0 ? 0 : (size_t)n_k_tiles * (2 * 128 * 128 + 128) * sizeof(float);
}

int fa_fwd_kvcache(const fa_tensor* q, const fa_tensor* k_cache, const fa_tensor* v_cache,
                   const fa_tensor* k_new, const fa_tensor* v_new, const fa_tensor* out,
                   const fa_tensor* lse, const fa_tensor* cu_seqlens_q,
                   const fa_tensor* cache_seqlens, const fa_tensor* block_table,
                   int32_t window_left, int32_t window_right, float softcap, float scale,
                   int32_t causal, int32_t append, const fa_opts* opts) {
  Plan pl;
  const KvNew kn{k_new, v_new, cache_seqlens, append};
  int rc = make_plan(q, k_cache, v_cache, out, lse, cu_seqlens_q, nullptr, block_table, nullptr, window_left,
                     window_right, softcap, scale, causal, opts, &pl, &kn);
  if (rc != FA_OK) return rc;
  return run_plan(pl, opts);
}

int fa_fwd_kvcache_plan(const fa_tensor* q, const fa_tensor* k_cache, const fa_tensor* v_cache,
                        const fa_tensor* k_new, const fa_tensor* v_new, const fa_tensor* out,
                        const fa_tensor* lse, const fa_tensor* cu_seqlens_q,
                        const fa_tensor* cache_seqlens, const fa_tensor* block_table,
                        int32_t window_left, int32_t window_right, float softcap, float scale,
                        int32_t causal, int32_t append, const fa_opts* opts, fa_plan* plan_out) {
  Plan pl;
  const KvNew kn{k_new, v_new, cache_seqlens, append};
  int rc = make_plan(q, k_cache, v_cache, out, lse, cu_seqlens_q, nullptr, block_table, nullptr, window_left,
                     window_right, softcap, scale, causal, opts, &pl, &kn);
  if (rc == FA_OK && plan_out) *plan_out = pl.pub;
  return rc;
}

}  // extern "C"

thread_local bool mfa::g_trace_ranges = true;

namespace {

// NVTX range around the host-side enqueue of one stage (a profiler's trace
// shows it beside the stage's kernels); none while g_trace_ranges is off.
struct TraceRange {
  bool on;
  explicit TraceRange(const char* name) : on(mfa::g_trace_ranges) {
    if (on) nvtxRangePushA(name);
  }
  ~TraceRange() {
    if (on) nvtxRangePop();
  }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

// Bind the workspace and enqueue a validated plan's kernels on opts->stream.
int run_plan(Plan& pl, const fa_opts* opts) {
  TraceRange tr_call("mfa.fwd");
  int rc;
  if (!opts->workspace || (reinterpret_cast<uintptr_t>(opts->workspace) % kAlign) != 0 ||
      opts->workspace_bytes < pl.pub.workspace_bytes)
    return FA_ERR_WORKSPACE;
  if ((rc = check_device()) != FA_OK) return rc;
  bind_workspace(&pl, opts->workspace);
  cudaStream_t st = static_cast<cudaStream_t>(opts->stream);
  const Params& P = pl.prm;
  // the counters are accumulated by the scheduler kernels, or written whole by
  // the prefill kernel when it schedules inline
  if ((!P.sched_inline || P.n_items == 0) && cudaMemsetAsync(P.stats, 0, 3 * sizeof(long long), st) != cudaSuccess)
    return FA_ERR_CUDA;
  if (P.n_items == 0) return FA_OK;
  cudaError_t e = cudaSuccess;
  if (!P.sched_inline) {
    if (P.mask_kind == FA_MASK_DENSE) {
      TraceRange tr("mfa.mask_summary");
      e = launch_mask_summary(P, st);
    }
    if (e == cudaSuccess && P.mask_kind == FA_MASK_TOPK) {
      TraceRange tr("mfa.topk_prep");
      e = launch_topk_prep(P, st);
    }
    // on the many-row path the top-k preparation has listed each unit's keys
    const bool listed = P.mask_kind == FA_MASK_TOPK && P.path == FA_PATH_PREFILL;
    if (e == cudaSuccess && !listed) {
      TraceRange tr("mfa.classify");
      e = launch_classify(P, st);
    }
  }
  cudaEvent_t ev_begin = static_cast<cudaEvent_t>(opts->event_begin);
  cudaEvent_t ev_attn_end = static_cast<cudaEvent_t>(opts->event_attn_end);
  if (e == cudaSuccess) {
    TraceRange tr(P.path == FA_PATH_PREFILL ? "mfa.prefill" : "mfa.decode");
    if (P.path == FA_PATH_PREFILL) {
      e = launch_prefill(P, st, ev_begin);
      if (e == cudaSuccess && ev_attn_end) e = cudaEventRecord(ev_attn_end, st);
    } else {
      e = launch_decode(P, st, ev_begin, ev_attn_end);
    }
  }
  if (e == cudaSuccess && opts->event_end)
    e = cudaEventRecord(static_cast<cudaEvent_t>(opts->event_end), st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_bwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
           const fa_tensor* lse, const fa_tensor* dout, const fa_tensor* dq, const fa_tensor* dk,
           const fa_tensor* dv, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
           int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
           const fa_opts* opts) {
  Plan pl;
  size_t off_delta = 0;
  int rc = make_plan_bwd(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, window_left,
                         window_right, softcap, scale, causal, opts, &pl, &off_delta);
  if (rc != FA_OK) return rc;
  if (!opts->workspace || (reinterpret_cast<uintptr_t>(opts->workspace) % kAlign) != 0 ||
      opts->workspace_bytes < pl.pub.workspace_bytes)
    return FA_ERR_WORKSPACE;
  if ((rc = check_device()) != FA_OK) return rc;
  bind_workspace(&pl, opts->workspace);
  Params& P = pl.prm;
  P.delta = reinterpret_cast<float*>(static_cast<unsigned char*>(opts->workspace) + off_delta);
  cudaStream_t st = static_cast<cudaStream_t>(opts->stream);
  TraceRange tr("mfa.bwd");
  cudaError_t e = launch_backward(P, st, static_cast<cudaEvent_t>(opts->event_begin));
  if (e == cudaSuccess && opts->event_end) e = cudaEventRecord(static_cast<cudaEvent_t>(opts->event_end), st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_bwd_plan(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                const fa_tensor* lse, const fa_tensor* dout, const fa_tensor* dq, const fa_tensor* dk,
                const fa_tensor* dv, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
                const fa_opts* opts, fa_plan* plan_out) {
  Plan pl;
  size_t off_delta = 0;
  int rc = make_plan_bwd(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, window_left,
                         window_right, softcap, scale, causal, opts, &pl, &off_delta);
  if (rc == FA_OK && plan_out) *plan_out = pl.pub;
  return rc;
}

int fa_check_device_error(void* stream, void* workspace, uint32_t* info) {
  if (!workspace) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader h;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (h.error != 0) {
    // the header and the tail-split counts, which an aborted launch may have left set
    unsigned char z[kWsHeadBytes];
    memset(z, 0, sizeof(z));
    if (cudaMemcpy(workspace, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (info) *info = h.error_info;
  return (int)h.error;
}

}  // extern "C"
