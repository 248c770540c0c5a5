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
//   3. topk_expiry: one warp per 128 consecutive ranks (eight warps per CTA
//      sharing the ranks in shared memory); F(t) for its ranks by a sweep over
//      a bitmap of the indices {S[0 .. t - 1]}: when S[t] falls below the
//      current F, it enters the K smallest and F moves down to the next index
//      present below it;
//   4. topk_gather (many-row path): per (sequence, head, 128-row query
//      tile) the list of every key some row of the tile keeps -- about
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
  constexpr int kPer = kRunKeys / kRunThreads;  // words per thread and run
  for (int o = 0; o < n_runs; ++o) {              // kPer loads in flight per thread
    uint64_t v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = src[o * kRunKeys + u * kRunThreads + threadIdx.x];
#pragma unroll
    for (int u = 0; u < kPer; ++u) runs[o * kRunKeys + u * kRunThreads + threadIdx.x] = v[u];
  }
  __syncthreads();
  int32_t* S = p.topk_rank + (int64_t)bh * p.Sk;
  int32_t* rho = p.topk_rho + (int64_t)bh * p.Sk;
  // this thread's words: place in its run plus, in every other run, the
  // number of words below it (a branch-free binary search over the run's
  // 2048 words; the kPer searches of a thread advance together)
  uint64_t w[kPer];
  int r[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    r[u] = u * kRunThreads + threadIdx.x;
    w[u] = runs[run * kRunKeys + r[u]];
  }
  for (int o = 0; o < n_runs; ++o) {
    if (o == run) continue;
    const uint64_t* R = runs + o * kRunKeys;
    int base[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) base[u] = 0;
#pragma unroll
    for (int step = kRunKeys / 2; step > 0; step >>= 1) {
#pragma unroll
      for (int u = 0; u < kPer; ++u)
        if (R[base[u] + step - 1] < w[u]) base[u] += step;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) r[u] += base[u] + (R[base[u]] < w[u] ? 1 : 0);
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (w[u] == ~0ull) continue;  // padding
    const int j = (int)(uint32_t)w[u];
    rho[j] = r[u];
    S[r[u]] = j;
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

// One CTA per (sequence, head) and group of kExpWarps chunks of kChunk ranks;
// the ranks rho are staged once per CTA as 16-bit values (Sk <= 16384).
// Each warp builds the bitmap of {S[0 .. t_lo - 1]} (index x is in it iff
// rho[x] < t_lo) from shared memory, finds F(t_lo) by counting, and one lane
// sweeps the chunk's ranks in order.
constexpr int kExpWarps = 8;

size_t expiry_smem(int n) {
  const int nw = (n + 31) / 32;
  return (size_t)nw * 64 + (size_t)kExpWarps * nw * 4 + (size_t)2 * kExpWarps * kChunk * 4;
}

__global__ void __launch_bounds__(32 * kExpWarps) topk_expiry_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char esm[];
  const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.Sk, K = p.keep_window, off = p.Sk - p.Sq;  // top-k takes fixed-length batches
  const int nw = (n + 31) >> 5;                                // bitmap words
  uint16_t* rho16 = reinterpret_cast<uint16_t*>(esm);         // [nw * 32], padding 0xffff
  uint32_t* bm = reinterpret_cast<uint32_t*>(esm + (size_t)nw * 64) + warp * nw;
  int* ys = reinterpret_cast<int*>(esm + (size_t)nw * 64 + (size_t)kExpWarps * nw * 4) + warp * kChunk;
  int* evs = ys + kExpWarps * kChunk;
  const int32_t* S = p.topk_rank + (int64_t)bh * n;
  const int32_t* rho = p.topk_rho + (int64_t)bh * n;
  int32_t* e = p.topk_e + (int64_t)bh * n;
  const int t_lo = (blockIdx.x * kExpWarps + warp) * kChunk, t_hi = min(t_lo + kChunk, n);
  const int cta_hi = min((int)(blockIdx.x + 1) * kExpWarps * kChunk, n);
  if (p.causal && cta_hi > K) {  // some warp of the CTA sweeps
    for (int x0 = 0; x0 < nw * 32; x0 += 8 * 32 * kExpWarps) {  // eight loads in flight per thread
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = x0 + u * 32 * kExpWarps + (int)threadIdx.x;
        v[u] = x < n ? __ldg(rho + x) : 0xffff;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = x0 + u * 32 * kExpWarps + (int)threadIdx.x;
        if (x < nw * 32) rho16[x] = (uint16_t)v[u];
      }
    }
    __syncthreads();
  }
  if (t_lo >= n) return;
  const int len = t_hi - t_lo;
  if (!p.causal || t_hi <= K) {
    // every row sees every key (kept set: the K best), or a rank below K:
    // fewer than K keys beat it anywhere
    for (int m = lane; m < len; m += 32) {
      const int t = t_lo + m;
      e[__ldg(S + t)] = (!p.causal && t >= K) ? kRowNever : kRowInf;
    }
    return;
  }
  for (int m = lane; m < len; m += 32) ys[m] = __ldg(S + t_lo + m);
  // the bitmap of {S[0 .. t_lo - 1]}: lane q reads ranks [8 q, 8 q + 8) and
  // four consecutive lanes assemble a word
  for (int q0 = 0; q0 < nw * 4; q0 += 32) {
    const int q = q0 + lane;
    unsigned b8 = 0;
    if (q < nw * 4) {
      const uint4 v = reinterpret_cast<const uint4*>(rho16)[q];
      const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        b8 |= ((int)(h[k] & 0xffffu) < t_lo ? 1u : 0u) << (2 * k);
        b8 |= ((int)(h[k] >> 16) < t_lo ? 1u : 0u) << (2 * k + 1);
      }
    }
    unsigned wv = b8 << (8 * (q & 3));
    wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
    if (q < nw * 4 && (q & 3) == 0) bm[q >> 2] = wv;
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
  // sweep: before rank t the set is {S[0 .. t - 1]}; a key entering below F
  // moves F down to the next index present below it (possibly itself)
  if (lane == 0) {
    int yn = ys[0];
    for (int m = 0; m < len; ++m) {
      const int t = t_lo + m, yt = yn;
      if (m + 1 < len) yn = ys[m + 1];
      if (t >= K) {
        evs[m] = F - off;
        if (yt < F) {
          bm[yt >> 5] |= 1u << (yt & 31);
          F = highest_below(bm, F);
        }
      } else {
        evs[m] = kRowInf;
        bm[yt >> 5] |= 1u << (yt & 31);
        if (t + 1 == K) F = highest_below(bm, n);  // the set holds exactly K keys: its largest index
      }
    }
  }
  __syncwarp();
  for (int m = lane; m < len; m += 32) e[ys[m]] = evs[m];
}

// 4 ------------------------------------------------------------------------
// Entry of a gathered key: x = key index | first row of the tile that keeps
// it << 16 | first row past the last one that does << 24 (rows relative to the
// tile, clamped to [0, 128]); y = its bias z * log2(e), as fp32 bits.
// One CTA per (sequence, head) and group of kListUnits units: the CTA of
// group x takes the row tiles x, x + GX, x + 2 GX, ... (GX groups), so that
// every CTA mixes short and long rows, and its warps work through the units
// one after the other, each warp on a contiguous share of the unit's keys
// (eight consecutive keys per lane and step).  The expiry rows e and the
// biases of the (sequence, head) are staged once in shared memory.  A first
// pass counts each warp's keys that every row of the tile keeps and the
// others; the second writes the entries, those keys first and the others
// after them, each group in key order (a prefix sum over the lanes and the
// warps' counts place them).  A key j every row of the tile may see (j <=
// r0 + off, or any key without the causal rule) is kept on rows [r0, e_j), so
// it is kept by some row iff e_j > r0 and by every row iff e_j > r1.
constexpr int kListWarps = 8;
constexpr int kListUnits = 8;

// e and z rows, each padded to a multiple of 8 entries (two 16-byte vector
// reads per lane and step), then per warp the entries of one step
size_t gather_smem(int n) { return (size_t)((n + 7) & ~7) * 8 + (size_t)kListWarps * 256 * 8; }

__global__ void __launch_bounds__(32 * kListWarps) topk_gather_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char gsm[];
  __shared__ int wcnt[kListWarps][4];  // per warp: keys every row keeps, the others, first of each kind
  const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.Sk, off = p.Sk - p.Sq;
  const int n8 = (n + 7) & ~7;
  int* es = reinterpret_cast<int*>(gsm);            // [n8] expiry rows
  float* zs = reinterpret_cast<float*>(gsm) + n8;   // [n8] biases, log2 units
  const int4* es4 = reinterpret_cast<const int4*>(es);
  const float4* zs4 = reinterpret_cast<const float4*>(zs);
  uint2* wbuf = reinterpret_cast<uint2*>(zs + n8) + warp * 256;  // this warp's entries of one step
  const int32_t* e = p.topk_e + (int64_t)bh * n;
  const float* z = z_row(p, bh);
  const int GX = gridDim.x;
  // keys some row of this CTA's units may see: [0, nks)
  int rt_max = blockIdx.x;
  for (int k = 1; k < kListUnits && rt_max + GX < p.n_row_tiles; ++k) rt_max += GX;
  const int nks = p.causal ? max(0, min(n, min(rt_max * 128 + 127, p.Sq - 1) + off + 1)) : n;
  // 16-byte loads when both rows allow them, else eight loads of each row in
  // flight per thread
  const bool vec = (n & 3) == 0 && p.z_sk == 1 && ((reinterpret_cast<uintptr_t>(e) | reinterpret_cast<uintptr_t>(z)) & 15) == 0;
  if (vec) {
    for (int x0 = 0; x0 < nks; x0 += 4 * 32 * kListWarps * 4) {
      int4 ev[4];
      float4 zv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int x = x0 + 4 * (u * 32 * kListWarps + (int)threadIdx.x);
        ev[u] = x < nks ? __ldg(reinterpret_cast<const int4*>(e + x)) : make_int4(0, 0, 0, 0);
        zv[u] = x < nks ? __ldg(reinterpret_cast<const float4*>(z + x)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int x = x0 + 4 * (u * 32 * kListWarps + (int)threadIdx.x);
        if (x < nks) {
          reinterpret_cast<int4*>(es)[x >> 2] = ev[u];
          reinterpret_cast<float4*>(zs)[x >> 2] =
              make_float4(zv[u].x * kLog2e, zv[u].y * kLog2e, zv[u].z * kLog2e, zv[u].w * kLog2e);
        }
      }
    }
  }
  for (int x0 = 0; !vec && x0 < nks; x0 += 8 * 32 * kListWarps) {
    int ev[8];
    float zv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int x = x0 + u * 32 * kListWarps + (int)threadIdx.x;
      ev[u] = x < nks ? __ldg(e + x) : 0;
      zv[u] = x < nks ? __ldg(z + (int64_t)x * p.z_sk) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int x = x0 + u * 32 * kListWarps + (int)threadIdx.x;
      if (x < nks) {
        es[x] = ev[u];
        zs[x] = zv[u] * kLog2e;
      }
    }
  }
  __syncthreads();
  unsigned long long n_f = 0, n_p = 0, n_e = 0;  // tile counts (thread 0)
  for (int k = 0; k < kListUnits; ++k) {
    const int rt = blockIdx.x + GX * k;
    if (rt >= p.n_row_tiles) break;
    const int r0 = rt * 128, r1 = min(r0 + 127, p.Sq - 1);
    const int64_t item = (int64_t)bh * p.n_row_tiles + rt;
    uint2* list = p.topk_list + item * ((int64_t)p.n_kt * kKeysPerTile);
    const int nk = p.causal ? max(0, min(n - 1, r1 + off) + 1) : n;  // keys some row may see: [0, nk)
    const int nb = p.causal ? max(0, min(nk, r0 + off + 1)) : nk;   // of those, seen by every row: [0, nb)
    const int steps = (nk + 255) >> 8, spw = (steps + kListWarps - 1) / kListWarps;
    const int s0 = warp * spw, s1 = min(s0 + spw, steps);
    // rows [a, c) of the tile keeping key j with expiry row ev
    auto rows = [&](int j, int ev, int& a, int& c) {
      a = j < nb ? r0 : max(j - off, r0);
      c = min(ev, r1 + 1);
    };
    int cf = 0, cp = 0, ff = INT_MAX, fk = INT_MAX;
    for (int st = s0; st < s1; ++st) {
      const int jl = st * 256 + 8 * lane;
      if (jl >= nk) continue;
      const int4 ea = es4[jl >> 2], eb = es4[(jl >> 2) + 1];
      const int ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
      if (jl + 8 <= nb) {  // every row may see these keys
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const bool full = ev[q] > r1, kept = ev[q] > r0;
          cf += full;
          cp += kept && !full;
          if (full) ff = min(ff, jl + q);
          if (kept) fk = min(fk, jl + q);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = jl + q;
          int a, c;
          rows(j, ev[q], a, c);
          const bool kept = j < nk && a < c, full = j < nk && a == r0 && c == r1 + 1;
          cf += full;
          cp += kept && !full;
          if (full) ff = min(ff, j);
          if (kept) fk = min(fk, j);
        }
      }
    }
    cf = (int)__reduce_add_sync(0xffffffffu, (unsigned)cf);
    cp = (int)__reduce_add_sync(0xffffffffu, (unsigned)cp);
    ff = __reduce_min_sync(0xffffffffu, ff);
    fk = __reduce_min_sync(0xffffffffu, fk);
    if (lane == 0) {
      wcnt[warp][0] = cf;
      wcnt[warp][1] = cp;
      wcnt[warp][2] = ff;
      wcnt[warp][3] = fk;
    }
    __syncthreads();
    int pos_f = 0, pos_p = 0, n_full = 0, n_part = 0, first_full = INT_MAX, first_kept = INT_MAX;
#pragma unroll
    for (int w = 0; w < kListWarps; ++w) {
      pos_f += w < warp ? wcnt[w][0] : 0;
      pos_p += w < warp ? wcnt[w][1] : 0;
      n_full += wcnt[w][0];
      n_part += wcnt[w][1];
      first_full = min(first_full, wcnt[w][2]);
      first_kept = min(first_kept, wcnt[w][3]);
    }
    // keys every row keeps first (so that whole tiles of them need no keep
    // test), then the others
    pos_p += n_full;
    for (int st = s0; st < s1; ++st) {
      const int jl = st * 256 + 8 * lane;
      const bool lane_in = jl < nk;
      int ev[8];
      float zv[8];
      {
        const int4 ea = lane_in ? es4[jl >> 2] : make_int4(0, 0, 0, 0);
        const int4 eb = lane_in ? es4[(jl >> 2) + 1] : make_int4(0, 0, 0, 0);
        const float4 za = lane_in ? zs4[jl >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 zb = lane_in ? zs4[(jl >> 2) + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
        ev[0] = ea.x; ev[1] = ea.y; ev[2] = ea.z; ev[3] = ea.w;
        ev[4] = eb.x; ev[5] = eb.y; ev[6] = eb.z; ev[7] = eb.w;
        zv[0] = za.x; zv[1] = za.y; zv[2] = za.z; zv[3] = za.w;
        zv[4] = zb.x; zv[5] = zb.y; zv[6] = zb.z; zv[7] = zb.w;
      }
      unsigned fl = 0, pl = 0;
      if (jl + 8 <= nb) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          fl |= (ev[q] > r1 ? 1u : 0u) << q;
          pl |= (ev[q] > r0 && ev[q] <= r1 ? 1u : 0u) << q;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = jl + q;
          int a, c;
          rows(j, ev[q], a, c);
          const bool in = j < nk, full = in && a == r0 && c == r1 + 1;
          fl |= (full ? 1u : 0u) << q;
          pl |= (in && a < c && !full ? 1u : 0u) << q;
        }
      }
      // entries before this lane's in the warp's share: an inclusive prefix
      // over the lanes of (keys every row keeps) | (the others) << 16
      const int cnt = __popc(fl) | (__popc(pl) << 16);
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
      }
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      const int tf = tot & 0xffff, tp = tot >> 16;
      // the step's entries go to the warp's buffer (those every row keeps,
      // then the others), then out to the list as two contiguous runs
      int wf = (inc - cnt) & 0xffff, wp = tf + ((inc - cnt) >> 16);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!(((fl | pl) >> q) & 1u)) continue;
        const int j = jl + q;
        int a, c;
        rows(j, ev[q], a, c);
        wbuf[((fl >> q) & 1u) ? wf++ : wp++] =
            make_uint2((uint32_t)j | ((uint32_t)(a - r0) << 16) | ((uint32_t)(c - r0) << 24), __float_as_uint(zv[q]));
      }
      __syncwarp();
      for (int i = lane; i < tf; i += 32) list[pos_f + i] = wbuf[i];
      for (int i = lane; i < tp; i += 32) list[pos_p + i] = wbuf[tf + i];
      __syncwarp();  // the buffer is read before the next step fills it
      pos_f += tf;
      pos_p += tp;
    }
    const int n_keys = n_full + n_part;
    // pad the last tile with a key no row keeps (a real key: its K/V rows are
    // finite, so P = 0 contributes exactly 0): the list's first key
    const int tiles = (n_keys + kKeysPerTile - 1) / kKeysPerTile;
    const uint32_t first_j = (uint32_t)(n_full > 0 ? first_full : first_kept);
    for (int i = n_keys + threadIdx.x; i < tiles * kKeysPerTile; i += blockDim.x)
      list[i] = make_uint2(first_j | (128u << 16), 0u);
    // the work list: gathered tile t, FULL for the leading tiles of keys every
    // row keeps, PARTIAL after them
    for (int t = threadIdx.x; t < tiles; t += blockDim.x)
      p.item_tiles[item * p.n_kt + t] = (t << 1) | (t >= n_full / kKeysPerTile ? 1 : 0);
    if (threadIdx.x == 0) {
      p.item_count[item] = tiles;
      p.topk_full[item] = n_full / kKeysPerTile;  // leading tiles of keys every row keeps
      n_f += n_full / kKeysPerTile;
      n_p += tiles - n_full / kKeysPerTile;
      n_e += (n + kKeysPerTile - 1) / kKeysPerTile - tiles;
    }
    __syncthreads();  // the warps' counts are read before the next unit writes them
  }
  if (threadIdx.x == 0) {
    atomicAdd(&p.stats[0], n_f);
    atomicAdd(&p.stats[1], n_p);
    atomicAdd(&p.stats[2], n_e);
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
  const int n_chunks = (p.Sk + kChunk - 1) / kChunk;
  const size_t esmem = expiry_smem(p.Sk);
  e = cudaFuncSetAttribute(topk_expiry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)esmem);
  if (e != cudaSuccess) return e;
  topk_expiry_kernel<<<dim3((n_chunks + kExpWarps - 1) / kExpWarps, bh), 32 * kExpWarps, esmem, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.path == FA_PATH_PREFILL) {
    const size_t gsmem = gather_smem(p.Sk);
    e = cudaFuncSetAttribute(topk_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsmem);
    if (e != cudaSuccess) return e;
    topk_gather_kernel<<<dim3((p.n_row_tiles + kListUnits - 1) / kListUnits, bh), 32 * kListWarps, gsmem, st>>>(p);
  } else {
    topk_tile_maxe_kernel<<<dim3(p.n_kt, bh), 128, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mfa
