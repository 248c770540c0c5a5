// sched.cu -- the tile scheduler: dense-mask summary, dynamic top-k preparation
// and (query-tile, key-tile) classification into FULL / PARTIAL / EMPTY.
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

// ---------------------------------------------------------------------------
// Dynamic top-k preparation.
//
// For a causal row i the candidates are keys 0..i+off; key j is kept while
// fewer than keep_window candidates beat it (larger z, or equal z and lower
// index).  Because the candidate set only grows with i, key j is kept exactly
// on rows [j - off, e_j), where e_j + off is the keep_window-th smallest index
// among the keys that beat j (never dropped if fewer than keep_window keys
// beat it).  Without the causal rule every row sees all keys, so the kept set
// is the global top keep_window.  Keys are compared as 64-bit words
// (order of z descending) << 32 | index, so "k beats j" is word_k < word_j.
// Two kernels compute e_j for every key:
//   1. topk_bucket_sort: one warp per bucket of 128 consecutive keys sorts the
//      bucket's words (bitonic network over registers and shuffles);
//   2. topk_expiry: one warp per key: each lane counts the beaters in up to
//      four buckets by binary search in their sorted words, a warp prefix sum
//      finds the bucket holding the keep_window-th beater, and ballots over
//      that bucket's keys, in index order, find its exact index.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_desc(float f) {
  if (f == 0.f) f = 0.f;  // -0 and +0 tie
  uint32_t u = __float_as_uint(f);
  u ^= (u & 0x80000000u) ? 0xffffffffu : 0x80000000u;  // ascending order of floats
  return ~u;                                             // descending
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}

// Sorted words of every bucket, one warp per bucket, 4 words per lane
// (element e = 4 lane + k); buckets past the end are padded with ~0.
__global__ void __launch_bounds__(256) topk_bucket_sort_kernel(const Params p) {
  const int bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  const int n = p.Sk;
  const int nb = (n + kKeysPerTile - 1) / kKeysPerTile;
  if (c >= nb) return;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const float* z = p.z + (int64_t)b * p.z_sb + (int64_t)h * p.z_sh;
  uint64_t v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = c * kKeysPerTile + 4 * lane + k;
    const float zj = j < n ? __ldg(z + (int64_t)j * p.z_sk) : 0.f;
    if ((p.debug_flags & FA_DEBUG_VALIDATE) && !isfinite(zj)) record_error(p, FA_ERR_DEVICE_VALUE, (uint32_t)c);
    v[k] = j < n ? (((uint64_t)ordered_desc(zj) << 32) | (uint32_t)j) : ~0ull;
  }
#pragma unroll
  for (int size = 2; size <= 128; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 4) {
        const int lm = stride >> 2;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = 4 * lane + k;
          const uint64_t o = shfl_xor64(v[k], lm);
          const bool up = (e & size) == 0;
          const bool lower = (e & stride) == 0;
          const uint64_t mn = v[k] < o ? v[k] : o, mx = v[k] < o ? o : v[k];
          v[k] = (lower == up) ? mn : mx;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if ((k & stride) == 0) {
            const int e = 4 * lane + k;
            const bool up = (e & size) == 0;
            const uint64_t x = v[k], y = v[k + stride];
            const bool swap = up ? (x > y) : (x < y);
            v[k] = swap ? y : x;
            v[k + stride] = swap ? x : y;
          }
        }
      }
    }
  }
  uint64_t* out = p.topk_sorted + (int64_t)bh * nb * kKeysPerTile + (int64_t)c * kKeysPerTile;
#pragma unroll
  for (int k = 0; k < 4; ++k) out[4 * lane + k] = v[k];
}

constexpr int kExpiryKeys = 256;   // keys per topk_expiry block (two key tiles)
constexpr int kBucketPad = 129;    // smem stride of a bucket's sorted words (bank spread)

__global__ void __launch_bounds__(256) topk_expiry_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int n = p.Sk;
  const int nb = (n + kKeysPerTile - 1) / kKeysPerTile;
  uint64_t* S = reinterpret_cast<uint64_t*>(smem);          // [nb][kBucketPad]
  uint32_t* zo = reinterpret_cast<uint32_t*>(S + (size_t)nb * kBucketPad);  // [nb * 128] ordered z
  __shared__ int e_s[kExpiryKeys];
  const int bh = blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int j_base = blockIdx.x * kExpiryKeys;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t* sorted = p.topk_sorted + (int64_t)bh * nb * kKeysPerTile;
  const float* z = p.z + (int64_t)b * p.z_sb + (int64_t)h * p.z_sh;
  for (int i = tid; i < nb * kKeysPerTile; i += blockDim.x) {
    S[(i / kKeysPerTile) * kBucketPad + (i % kKeysPerTile)] = __ldg(sorted + i);
    zo[i] = i < n ? ordered_desc(__ldg(z + (int64_t)i * p.z_sk)) : 0xffffffffu;
  }
  __syncthreads();
  const int W = p.keep_window;
  const int off = p.Sk - p.Sq;  // top-k needs a fixed-length batch
  int32_t* e_out = p.topk_e + (int64_t)bh * n;
  for (int q = 0; q < kExpiryKeys / 8; ++q) {
    const int jl = warp * (kExpiryKeys / 8) + q;
    const int j = j_base + jl;
    if (j >= n) break;
    const uint64_t wj = ((uint64_t)zo[j] << 32) | (uint32_t)j;
    // beaters of j in buckets lane + 32 s (s = 0..3: up to 128 buckets)
    constexpr int kSeg = kMaxTopkKeys / kKeysPerTile / 32;
    int cnt[kSeg], inc[kSeg];
#pragma unroll
    for (int sg = 0; sg < kSeg; ++sg) {
      const int c = lane + 32 * sg;
      int lo = 0;
      if (c < nb) {
        const uint64_t* Sc = S + c * kBucketPad;
        int hi = kKeysPerTile;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (Sc[mid] < wj) lo = mid + 1; else hi = mid;
        }
      }
      cnt[sg] = lo;
      inc[sg] = lo;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int sg = 0; sg < kSeg; ++sg) {
        const int a = __shfl_up_sync(0xffffffffu, inc[sg], o);
        if (lane >= o) inc[sg] += a;
      }
    }
#pragma unroll
    for (int sg = 1; sg < kSeg; ++sg) inc[sg] += __shfl_sync(0xffffffffu, inc[sg - 1], 31);
    const int total = __shfl_sync(0xffffffffu, inc[kSeg - 1], 31);
    int e;
    if (total < W) {
      e = kRowInf;   // fewer than keep_window keys beat j anywhere
    } else if (!p.causal) {
      e = kRowNever;
    } else {
      int c = -1, need = 0;
#pragma unroll
      for (int sg = 0; sg < kSeg; ++sg) {
        const unsigned hit = __ballot_sync(0xffffffffu, inc[sg] >= W);
        if (c < 0 && hit) {
          const int l = __ffs(hit) - 1;
          c = l + 32 * sg;
          need = W - (__shfl_sync(0xffffffffu, inc[sg], l) - __shfl_sync(0xffffffffu, cnt[sg], l));
        }
      }
      // the need-th beater of j in bucket c, in index order
      int bw = n;
      const int c0 = c * kKeysPerTile;
#pragma unroll
      for (int i = 0; i < kKeysPerTile / 32; ++i) {
        const int jj = c0 + 32 * i + lane;
        const bool beats = jj < n && ((((uint64_t)zo[jj] << 32) | (uint32_t)jj) < wj);
        const unsigned m = __ballot_sync(0xffffffffu, beats);
        const int pc = __popc(m);
        if (need <= pc) {
          bw = c0 + 32 * i + (int)__fns(m, 0, need);
          break;
        }
        need -= pc;
      }
      e = bw - off;
    }
    if (lane == 0) {
      e_out[j] = e;
      e_s[jl] = e;
    }
  }
  __syncthreads();
  // per key tile: the largest e (a tile is dead for rows >= max e)
  if (warp < kExpiryKeys / kKeysPerTile) {
    const int kt = (j_base / kKeysPerTile) + warp;
    const int j0 = kt * kKeysPerTile;
    if (j0 < n) {
      int mx = kRowNever;
      for (int jj = lane; jj < kKeysPerTile && j0 + jj < n; jj += 32) mx = max(mx, e_s[warp * kKeysPerTile + jj]);
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) p.topk_tile_maxe[(int64_t)bh * p.n_kt + kt] = mx;
    }
  }
}

size_t topk_expiry_smem(int Sk) {
  const size_t nb = (Sk + kKeysPerTile - 1) / kKeysPerTile;
  return nb * kBucketPad * 8 + nb * kKeysPerTile * 4;
}

cudaError_t launch_topk_prep(const Params& p, cudaStream_t st) {
  const int nb = (p.Sk + kKeysPerTile - 1) / kKeysPerTile;
  dim3 g1((nb + 7) / 8, p.n_seq * p.Hq);
  topk_bucket_sort_kernel<<<g1, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem2 = topk_expiry_smem(p.Sk);
  e = cudaFuncSetAttribute(topk_expiry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  if (e != cudaSuccess) return e;
  dim3 g2((p.Sk + kExpiryKeys - 1) / kExpiryKeys, p.n_seq * p.Hq);
  topk_expiry_kernel<<<g2, 256, smem2, st>>>(p);
  return cudaGetLastError();
}

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
