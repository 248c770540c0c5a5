// topk.cu -- preparation of the dynamic top-k mask of flash-sparse-attention
// issue 11, "[Integration Progress Report] Dynamic Mask Attention Integration
// into FlashAttention" ("Overview": Python precomputes zero_hold_states; the
// CUDA mask does causal masking and top-k selection).
//
// For a causal row i the candidates are keys 0 .. i + off; key j is kept
// while fewer than keep_window (K) candidates beat it (larger z, or equal z and
// lower index).  The candidate set only grows with i, so key j is kept exactly
// on rows [j - off, e_j).  Rank the keys from best to worst (S[t] = key of rank
// t, rho[j] = rank of key j): the keys that beat j are S[0 .. rho[j] - 1], so
// e_j + off is the K-th smallest index among them, F(rho[j]), with
// F(t) = K-th smallest index of {S[0], ..., S[t - 1]}; a key of rank < K is
// never dropped.  Without the causal rule every row sees every key and the
// kept set is the K best.
//
// Kernels (one launch each, all on the caller's stream):
//   1. topk_sort_runs: one CTA sorts a run of 2048 keys of one (sequence,
//      head) by the word (z order, descending) << 32 | index (bitonic network
//      in shared memory);
//   2. topk_rank: each key's rank = its place in its run plus, for every other
//      run, the number of words below it there (binary search); writes rho and S;
//   3. topk_expiry: one warp per 128 consecutive ranks; F(t) for its ranks by
//      a sweep over a bitmap of the indices {S[0 .. t - 1]}: when S[t] falls
//      below the current F, it enters the K smallest and F moves down to the
//      next index present below it;
//   4. topk_gather (many-row path): one CTA per (sequence, head, 128-row
//      query tile) lists every key some row of the tile keeps -- about
//      keep_window of them instead of every causally allowed key -- with the
//      rows of the tile that keep it and its bias: first the keys every row
//      keeps, then the others, each group in key order; the attention kernel
//      fetches exactly these keys (TMA gather) as dense 128-key tiles, and the
//      tiles made only of keys every row keeps need no keep test (FULL);
//   5. topk_tile_maxe (few-row path): per 128-key tile, the largest e_j, so
//      that the scheduler can drop tiles no row keeps any key of.
#include <cuda_runtime.h>

#include <climits>

#include "fa_device.cuh"

namespace mfa {

namespace {

constexpr int kRunKeys = 2048;     // keys per sorted run (one CTA)
constexpr int kRunThreads = 256;
constexpr int kMaxRuns = kMaxTopkKeys / kRunKeys;
constexpr int kChunk = 128;        // ranks per topk_expiry warp
constexpr int kMaxWords = kMaxTopkKeys / 32;

__device__ __forceinline__ uint32_t ordered_desc(float f) {
  if (f == 0.f) f = 0.f;  // -0 and +0 tie
  uint32_t u = __float_as_uint(f);
  u ^= (u & 0x80000000u) ? 0xffffffffu : 0x80000000u;  // ascending order of floats
  return ~u;                                             // descending
}

__device__ __forceinline__ const float* z_row(const Params& p, int bh) {
  return p.z + (int64_t)(bh / p.Hq) * p.z_sb + (int64_t)(bh % p.Hq) * p.z_sh;
}

// 1 ------------------------------------------------------------------------
__global__ void __launch_bounds__(kRunThreads) topk_sort_runs_kernel(const Params p) {
  __shared__ uint64_t s[kRunKeys];
  const int run = blockIdx.x, bh = blockIdx.y;
  const float* z = z_row(p, bh);
  const int j0 = run * kRunKeys;
  for (int i = threadIdx.x; i < kRunKeys; i += kRunThreads) {
    const int j = j0 + i;
    uint64_t w = ~0ull;  // padding sorts last
    if (j < p.Sk) {
      const float zj = __ldg(z + (int64_t)j * p.z_sk);
      if ((p.debug_flags & FA_DEBUG_VALIDATE) && !isfinite(zj)) record_error(p, FA_ERR_DEVICE_VALUE, (uint32_t)j);
      w = ((uint64_t)ordered_desc(zj) << 32) | (uint32_t)j;
    }
    s[i] = w;
  }
  __syncthreads();
  // Bitonic network, ascending.  Pair t joins element i = 2t - (t mod j) with
  // i + j; for j <= 32 the 64 elements [64 m, 64 m + 64) are handled by warp
  // m mod 8 alone, so consecutive such stages need only a warp barrier.
  for (int k = 2; k <= kRunKeys; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = threadIdx.x; t < kRunKeys / 2; t += kRunThreads) {
        const int i = 2 * t - (t & (j - 1)), l = i + j;
        const bool up = (i & k) == 0;
        const uint64_t a = s[i], c = s[l];
        if ((a > c) == up) {
          s[i] = c;
          s[l] = a;
        }
      }
      const int next_j = j > 1 ? j >> 1 : k;  // first stride of the next size
      if (j <= 32 && next_j <= 32) __syncwarp(); else __syncthreads();
    }
  }
  uint64_t* out = p.topk_runs + ((int64_t)bh * gridDim.x + run) * kRunKeys;
  for (int i = threadIdx.x; i < kRunKeys; i += kRunThreads) out[i] = s[i];
}

// 2 ------------------------------------------------------------------------
__global__ void __launch_bounds__(kRunThreads) topk_rank_kernel(const Params p) {
  extern __shared__ uint64_t runs[];  // [n_runs][kRunKeys]
  const int run = blockIdx.x, n_runs = gridDim.x, bh = blockIdx.y;
  const uint64_t* src = p.topk_runs + (int64_t)bh * n_runs * kRunKeys;
  for (int i = threadIdx.x; i < n_runs * kRunKeys; i += kRunThreads) runs[i] = src[i];
  __syncthreads();
  int32_t* S = p.topk_rank + (int64_t)bh * p.Sk;
  int32_t* rho = p.topk_rho + (int64_t)bh * p.Sk;
  for (int i = threadIdx.x; i < kRunKeys; i += kRunThreads) {
    const uint64_t w = runs[run * kRunKeys + i];
    if (w == ~0ull) continue;  // padding
    int r = i;
    for (int o = 0; o < n_runs; ++o) {
      if (o == run) continue;
      const uint64_t* R = runs + o * kRunKeys;
      int lo = 0, hi = kRunKeys;  // words below w (words are distinct; padding is never below)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (R[mid] < w) lo = mid + 1; else hi = mid;
      }
      r += lo;
    }
    const int j = (int)(uint32_t)w;
    rho[j] = r;
    S[r] = j;
  }
}

// 3 ------------------------------------------------------------------------
// Bitmap helpers over the indices [0, n): word w of the set in bm[w].
__device__ __forceinline__ int highest_below(const uint32_t* bm, int F) {
  int wi = F >> 5;
  uint32_t m = (F & 31) ? (bm[wi] & ((1u << (F & 31)) - 1u)) : 0u;
  while (!m && wi > 0) m = bm[--wi];
  return m ? wi * 32 + 31 - __clz((int)m) : -1;
}

__global__ void __launch_bounds__(32) topk_expiry_kernel(const Params p) {
  __shared__ uint32_t bm[kMaxWords];
  const int bh = blockIdx.y, lane = threadIdx.x;
  const int n = p.Sk, K = p.keep_window, off = p.Sk - p.Sq;  // top-k takes fixed-length batches
  const int t_lo = blockIdx.x * kChunk, t_hi = min(t_lo + kChunk, n);
  const int32_t* S = p.topk_rank + (int64_t)bh * n;
  const int32_t* rho = p.topk_rho + (int64_t)bh * n;
  int32_t* e = p.topk_e + (int64_t)bh * n;
  int y[kChunk / 32];  // S[t] for the chunk's ranks t = t_lo + 32 m + lane
  int ev[kChunk / 32];
#pragma unroll
  for (int m = 0; m < kChunk / 32; ++m) {
    const int t = t_lo + 32 * m + lane;
    y[m] = t < t_hi ? S[t] : 0;
    ev[m] = kRowInf;  // rank < K: fewer than K keys beat it anywhere
  }
  if (!p.causal) {
#pragma unroll
    for (int m = 0; m < kChunk / 32; ++m) {
      const int t = t_lo + 32 * m + lane;
      if (t < t_hi) e[y[m]] = t < K ? kRowInf : kRowNever;
    }
    return;
  }
  if (t_hi > K) {
    // the set {S[0 .. t_lo - 1]}: index x is in it iff rho[x] < t_lo
    const int nw = (n + 31) >> 5;
    for (int w0 = 0; w0 < nw; w0 += 8) {  // eight words' loads in flight at a time
      bool in[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = 32 * (w0 + u) + lane;
        in[u] = x < n && __ldg(rho + x) < t_lo;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const unsigned bits = __ballot_sync(0xffffffffu, in[u]);
        if (lane == 0 && w0 + u < nw) bm[w0 + u] = bits;
      }
    }
    __syncwarp();
    int F = -1;
    if (t_lo >= K) {
      // the K-th smallest index present: words counted in lane-contiguous blocks
      const int wpl = (nw + 31) >> 5;
      int c = 0;
      for (int w = lane * wpl; w < min(nw, lane * wpl + wpl); ++w) c += __popc(bm[w]);
      int inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += a;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, inc >= K);
      const int L = __ffs(hit) - 1;  // t_lo >= K guarantees a hit
      int need = K - (__shfl_sync(0xffffffffu, inc, L) - __shfl_sync(0xffffffffu, c, L));
      if (lane == L) {
        for (int w = L * wpl;; ++w) {
          const int pc = __popc(bm[w]);
          if (need <= pc) {
            F = 32 * w + (int)__fns(bm[w], 0, need);
            break;
          }
          need -= pc;
        }
      }
      F = __shfl_sync(0xffffffffu, F, L);
    }
    // sweep: before rank t the set is {S[0 .. t - 1]}
    for (int t = t_lo; t < t_hi; ++t) {
      const int m = (t - t_lo) >> 5;
      int yt = 0;
#pragma unroll
      for (int mm = 0; mm < kChunk / 32; ++mm)
        if (mm == m) yt = __shfl_sync(0xffffffffu, y[mm], (t - t_lo) & 31);
      if (t >= K) {
        if (lane == ((t - t_lo) & 31)) ev[m] = F - off;
        if (yt < F) {
          if (lane == 0) bm[yt >> 5] |= 1u << (yt & 31);
          __syncwarp();
          F = highest_below(bm, F);  // yt itself, or the next index present below F
        }
      } else {
        if (lane == 0) bm[yt >> 5] |= 1u << (yt & 31);
        __syncwarp();
        if (t + 1 == K) F = highest_below(bm, n);  // the set holds exactly K keys: its largest index
      }
      __syncwarp();
    }
  }
#pragma unroll
  for (int m = 0; m < kChunk / 32; ++m) {
    const int t = t_lo + 32 * m + lane;
    if (t < t_hi) e[y[m]] = ev[m];
  }
}

// 4 ------------------------------------------------------------------------
// Entry of a gathered key: x = key index | first row of the tile that keeps
// it << 16 | first row past the last one that does << 24 (rows relative to the
// tile, clamped to [0, 128]); y = its bias z * log2(e), as fp32 bits.
// One CTA per unit; thread t takes the keys [t * per, (t + 1) * per) (all its
// loads in flight at once), a block-wide scan of the threads' counts places
// its kept keys, so the list comes out in key order.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) topk_gather_kernel(const Params p) {
  __shared__ int wsum[kGatherThreads / 32];
  const int rt = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.Sk, off = p.Sk - p.Sq;
  const int r0 = rt * 128, r1 = min(r0 + 127, p.Sq - 1);
  const int64_t item = (int64_t)bh * p.n_row_tiles + rt;
  uint2* list = p.topk_list + item * ((int64_t)p.n_kt * kKeysPerTile);
  const int32_t* e = p.topk_e + (int64_t)bh * n;
  const float* z = z_row(p, bh);
  const int jmax = p.causal ? min(n - 1, r1 + off) : n - 1;
  const int per = (n + kGatherThreads - 1) / kGatherThreads;  // keys per thread (<= 64)
  const int ja = tid * per, jb = min(ja + per, jmax + 1);      // this thread's keys [ja, jb)
  // which of this thread's keys some row of the tile keeps (one bit each), and
  // of those, which every row of the tile keeps
  static_assert(kMaxTopkKeys / kGatherThreads <= 64, "one 64-bit mask per thread");
  uint64_t bits = 0, full = 0;
#pragma unroll 8
  for (int j = ja; j < jb; ++j) {
    // the tile's rows keeping key j are [a, c) (absolute rows; e_j may be
    // INT_MIN, so nothing is subtracted before the comparison)
    const int a = max(p.causal ? j - off : INT_MIN, r0);
    const int c = min(__ldg(e + j), r1 + 1);
    if (a < c) bits |= 1ull << (j - ja);
    if (a == r0 && c == r1 + 1) full |= 1ull << (j - ja);
  }
  // exclusive scan over the block of (keys every row keeps) | (the others) << 16
  const int cf = __popcll(full), cp = __popcll(bits & ~full);
  int inc = cf | (cp << 16);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kGatherThreads / 32; ++w) {
    before += (w < warp) ? wsum[w] : 0;
    total += wsum[w];
  }
  const int ex = before + inc - (cf | (cp << 16));
  const int n_full = total & 0xffff, n_keys = n_full + (total >> 16);
  // keys every row keeps first (so that whole tiles of them need no keep
  // test), then the others; each group in key order
  int pos_f = ex & 0xffff, pos_p = n_full + (ex >> 16);
  for (uint64_t m = bits; m; m &= m - 1) {
    const int q = __ffsll((long long)m) - 1, j = ja + q;
    const int lo = max(p.causal ? j - off : INT_MIN, r0) - r0;  // listed: 0 <= lo < hi <= 128
    const int hi = min(__ldg(e + j), r1 + 1) - r0;
    const uint2 ent = make_uint2((uint32_t)j | ((uint32_t)lo << 16) | ((uint32_t)hi << 24),
                                 __float_as_uint(__ldg(z + (int64_t)j * p.z_sk) * kLog2e));
    list[((full >> q) & 1) ? pos_f++ : pos_p++] = ent;
  }
  // pad the last tile with a key no row keeps (a real key: its K/V rows are
  // finite, so P = 0 contributes exactly 0); list[0] is a listed key
  const int tiles = (n_keys + kKeysPerTile - 1) / kKeysPerTile;
  __syncthreads();
  if (n_keys > 0) {
    const uint32_t first_j = list[0].x & 0xffffu;
    for (int i = n_keys + tid; i < tiles * kKeysPerTile; i += kGatherThreads)
      list[i] = make_uint2(first_j | (128u << 16), 0u);
  }
  // the work list: gathered tile t, FULL for the leading tiles of keys every
  // row keeps, PARTIAL after them
  for (int t = tid; t < tiles; t += kGatherThreads)
    p.item_tiles[item * p.n_kt + t] = (t << 1) | (t >= n_full / kKeysPerTile ? 1 : 0);
  if (tid == 0) {
    p.item_count[item] = tiles;
    p.topk_full[item] = n_full / kKeysPerTile;  // leading tiles of keys every row keeps
    const int n_kt_b = (n + kKeysPerTile - 1) / kKeysPerTile;
    atomicAdd(&p.stats[0], (unsigned long long)(n_full / kKeysPerTile));
    atomicAdd(&p.stats[1], (unsigned long long)(tiles - n_full / kKeysPerTile));
    atomicAdd(&p.stats[2], (unsigned long long)(n_kt_b - tiles));
  }
}

// 5 ------------------------------------------------------------------------
__global__ void __launch_bounds__(128) topk_tile_maxe_kernel(const Params p) {
  const int kt = blockIdx.x, bh = blockIdx.y;
  const int j = kt * kKeysPerTile + threadIdx.x;
  int v = j < p.Sk ? p.topk_e[(int64_t)bh * p.Sk + j] : kRowNever;
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __shared__ int wmax[4];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0)
    p.topk_tile_maxe[(int64_t)bh * p.n_kt + kt] = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
}

}  // namespace

int topk_n_runs(int Sk) { return (Sk + kRunKeys - 1) / kRunKeys; }

cudaError_t launch_topk_prep(const Params& p, cudaStream_t st) {
  const int n_runs = topk_n_runs(p.Sk);
  const int bh = p.n_seq * p.Hq;
  if (n_runs < 1 || n_runs > kMaxRuns || bh <= 0) return cudaErrorInvalidValue;
  topk_sort_runs_kernel<<<dim3(n_runs, bh), kRunThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int smem = n_runs * kRunKeys * 8;
  e = cudaFuncSetAttribute(topk_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_rank_kernel<<<dim3(n_runs, bh), kRunThreads, smem, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_expiry_kernel<<<dim3((p.Sk + kChunk - 1) / kChunk, bh), 32, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.path == FA_PATH_PREFILL) {
    topk_gather_kernel<<<dim3(p.n_row_tiles, bh), kGatherThreads, 0, st>>>(p);
  } else {
    topk_tile_maxe_kernel<<<dim3(p.n_kt, bh), 128, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mfa
