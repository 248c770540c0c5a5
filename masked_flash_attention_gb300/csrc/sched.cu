// sched.cu -- the tile scheduler: dense-mask summary and (query-tile, key-tile)
// classification into FULL / PARTIAL / EMPTY.
//
// EMPTY tiles (every pair masked) are left out of the work list, so no kernel
// ever computes them: the ExecuTorch pull request 10466 "Summary" notes that
// a chunk whose mask is entirely -inf could have been skipped outright.
#include <cuda_runtime.h>

#include "fa_device.cuh"

namespace mfa {

// ---------------------------------------------------------------------------
// Dense mask summary: one block per (mask batch, mask head, row tile, key tile)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) mask_summary_kernel(const Params p) {
  const int64_t blk = blockIdx.x;
  const int kt = (int)(blk % p.n_kt);
  int64_t t = blk / p.n_kt;
  const int rt = (int)(t % p.n_row_tiles);
  t /= p.n_row_tiles;
  const int mh = (int)(t % p.m_nh);
  const int mb = (int)(t / p.m_nh);
  int i0, i1;
  tile_rows(p, rt, i0, i1);
  i1 = min(i1, p.Sq - 1);
  const int kj0 = kt * kKeysPerTile;
  const int kj1 = min(kj0 + kKeysPerTile, p.Sk) - 1;
  const int nr = i1 - i0 + 1, nk = kj1 - kj0 + 1;
  bool any_nonneg = false, any_nonzero = false, any_bad = false;
  if (nr > 0 && nk > 0) {
    const float* base = p.mask + (int64_t)mb * p.m_sb + (int64_t)mh * p.m_sh;
    for (int e = threadIdx.x; e < nr * nk; e += blockDim.x) {
      int r = i0 + e / nk, j = kj0 + e % nk;
      float m = __ldg(base + (int64_t)r * p.m_sq + (int64_t)j * p.m_sk);
      any_nonneg |= (m != -INFINITY);
      any_nonzero |= (m != 0.f);
      any_bad |= !(m < INFINITY);  // NaN or +inf
    }
  }
  int nonneg = __syncthreads_or(any_nonneg);
  int nonzero = __syncthreads_or(any_nonzero);
  if ((p.debug_flags & FA_DEBUG_VALIDATE) && __syncthreads_or(any_bad) && threadIdx.x == 0)
    record_error(p, FA_ERR_DEVICE_VALUE, (uint32_t)blk);
  if (threadIdx.x == 0) {
    uint8_t cls = !nonneg ? kMaskEmpty : (!nonzero ? kMaskZero : kMaskMixed);
    p.mask_summary[blk] = cls;
  }
}

cudaError_t launch_mask_summary(const Params& p, cudaStream_t st) {
  int64_t n = (int64_t)p.m_nb * p.m_nh * p.n_row_tiles * p.n_kt;
  if (n <= 0) return cudaSuccess;
  mask_summary_kernel<<<(unsigned)n, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// The dynamic top-k preparation (expiry rows, tile summaries, gathered key
// lists) is in topk.cu.

// ---------------------------------------------------------------------------
// Classification: one warp per item (sequence, head, row tile).  Emits the
// ordered list of non-EMPTY key tiles, each flagged FULL or PARTIAL.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) classify_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (item >= p.n_items) return;
  const int rt = (int)(item % p.n_row_tiles);
  const int64_t t = item / p.n_row_tiles;
  const int hs = (int)(t % p.n_heads_sched);
  const int b = (int)(t / p.n_heads_sched);
  const int q_len = seq_qlen(p, b), kv_len = seq_klen(p, b);
  // the lengths come from device memory: check them against the sizes the
  // host planned for before anything indexes with them
  if (seq_lengths_bad(p, b, q_len, kv_len)) {
    if (lane == 0) {
      p.item_count[item] = -1;  // the attention kernels leave this item alone
      record_error(p, FA_ERR_DEVICE_BOUNDS, (uint32_t)b);
    }
    return;
  }
  const int off = kv_len - q_len;
  int i0, i1;
  tile_rows(p, rt, i0, i1);
  int32_t* out = p.item_tiles + item * p.n_kt;
  const int n_kt_b = (kv_len + kKeysPerTile - 1) / kKeysPerTile;
  if (i0 >= q_len || kv_len <= 0) {
    if (lane == 0) {
      p.item_count[item] = 0;
      if (i0 < q_len) atomicAdd(&p.stats[2], (unsigned long long)n_kt_b);
    }
    return;
  }
  i1 = min(i1, q_len - 1);
  // q-heads covered by this item (decode items pack a group's heads)
  int h_lo, h_hi;
  if (p.path == FA_PATH_DECODE) {
    h_lo = hs * p.G;
    h_hi = h_lo + p.G - 1;
  } else {
    h_lo = h_hi = hs;
  }
  const bool no_skip = (p.debug_flags & FA_DEBUG_NO_SKIP) != 0;
  int kt_lo = 0, kt_hi = n_kt_b - 1;
  if (!no_skip) {
    int jlo, jhi;
    key_range(p, i0, i1, off, kv_len, jlo, jhi);
    if (jlo > jhi) { kt_lo = 0; kt_hi = -1; }
    else { kt_lo = jlo / kKeysPerTile; kt_hi = jhi / kKeysPerTile; }
  }
  int count = 0;
  unsigned long long n_full = 0, n_part = 0;
  for (int base = kt_lo; base <= kt_hi; base += 32) {
    int kt = base + lane;
    bool live = kt <= kt_hi;
    bool partial = true;
    if (live && !no_skip) {
      int kj0 = kt * kKeysPerTile, kj1 = kj0 + kKeysPerTile - 1;
      partial = !tile_all_allowed(p, i0, i1, kj0, kj1, off, kv_len);
      if (p.mask_kind == FA_MASK_DENSE) {
        bool any_live = false, any_mixed = false;
        for (int h = h_lo; h <= h_hi; ++h) {
          int mb = p.m_nb > 1 ? b : 0, mh = p.m_nh > 1 ? h : 0;
          uint8_t c = p.mask_summary[(((int64_t)mb * p.m_nh + mh) * p.n_row_tiles + rt) * p.n_kt + kt];
          any_live |= (c != kMaskEmpty);
          any_mixed |= (c == kMaskMixed);
          if (p.m_nh == 1) break;
        }
        if (!any_live) live = false;
        partial |= any_mixed;
      } else if (p.mask_kind == FA_MASK_TOPK) {
        bool any_live = false;
        for (int h = h_lo; h <= h_hi; ++h) {
          int mx = p.topk_tile_maxe[((int64_t)b * p.Hq + h) * p.n_kt + kt];
          any_live |= (mx > i0);
        }
        if (!any_live) live = false;
        partial = true;  // the bias is added on every kept pair
      }
    }
    unsigned bal = __ballot_sync(0xffffffffu, live);
    if (live) {
      int pos = count + __popc(bal & ((1u << lane) - 1u));
      out[pos] = (kt << 1) | (partial ? 1 : 0);
      if (partial) ++n_part; else ++n_full;
    }
    count += __popc(bal);
  }
  for (int o = 16; o > 0; o >>= 1) {
    n_full += __shfl_xor_sync(0xffffffffu, n_full, o);
    n_part += __shfl_xor_sync(0xffffffffu, n_part, o);
  }
  if (lane == 0) {
    p.item_count[item] = count;
    atomicAdd(&p.stats[0], n_full);
    atomicAdd(&p.stats[1], n_part);
    atomicAdd(&p.stats[2], (unsigned long long)(n_kt_b - count));
  }
}

cudaError_t launch_classify(const Params& p, cudaStream_t st) {
  if (p.n_items <= 0) return cudaSuccess;
  int64_t blocks = (p.n_items + 7) / 8;
  classify_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mfa
