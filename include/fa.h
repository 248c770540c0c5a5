/*
 * fa.h -- C ABI of the GB300 (sm_103a) masked flash-attention forward library
 * (libmfa_gb300.so).
 *
 * One call, fa_fwd(), computes masked softmax attention
 *
 *     O[i] = sum_j softmax_j(x_ij) V[j],   LSE[i] = log sum_j exp(x_ij)
 *
 * with the logit x_ij built, in this order, from
 *   - the scaled dot product  scale * <Q[i], K[j]>;
 *   - the logit soft-cap  softcap * tanh(x / softcap)  when softcap > 0
 *     (the `softcap` argument of vLLM pull request 11277's
 *     flash_attn_varlen_func call);
 *   - pair rules that set x_ij = -inf: causal aligned bottom-right, i.e. the
 *     last query row sits on the last key, j <= i + (kv_len - q_len)
 *     (FastChat pull request 2315, "Optimize for proper flash attn causal
 *     handling": q_len != kv_len over past key-values without padding q);
 *     a sliding window j >= i + off - window_left, j <= i + off + window_right
 *     (`window_size` of the vLLM call; the ExecuTorch pull request 10466
 *     "Summary" builds the same window from an additive mask); j < kv_len;
 *   - an additive term added after the soft-cap: a dense fp32 mask M[i, j]
 *     whose -inf entries drop keys (ExecuTorch pull request 10466,
 *     "Summary"), or the dynamic top-k mask of flash-sparse-attention issue
 *     11 ("[Integration Progress Report] Dynamic Mask Attention Integration
 *     into FlashAttention", "Overview"): for each query row, among the keys
 *     the pair rules allow, only the keep_window keys with the largest
 *     zero_hold_states value are kept (ties: lower key index wins) and that
 *     value is added to their logit.
 * A query row with no kept key gets O = 0 and LSE = -inf, never NaN
 * (ExecuTorch pull request 10466, "Summary": a fully -inf chunk must not
 * poison the running softmax).
 *
 * Grouped-query heads: Hq must be a multiple of Hkv; q-head h reads K/V head
 * h / (Hq / Hkv); K/V are never expanded (InfiniTrain pull request 193, "feat:
 * Flash Attention", sections "Framework 与 autograd" and "Transformer 接入").
 *
 * Element type: q, k, v and out are all bf16 or all fp16 (the two input
 * types of the FlashAttention-2 kernels in InfiniTrain pull request 193,
 * "FlashAttention native backend"; "bf16" below stands for either).  Logits,
 * the softmax and the accumulators are fp32; P enters the PV product in the
 * input type; out is written in the input type.
 *
 * Layouts (element strides; the head-dim stride must be 1, every other stride
 * a multiple of 8 elements, every base pointer 16-byte aligned):
 *   q    bf16 [B, Sq, Hq, d]                      fixed-length batch
 *        bf16 [total_q, Hq, d]                    with cu_seqlens_q
 *   k, v bf16 [B, Sk, Hkv, d]                     fixed-length batch
 *        bf16 [total_k, Hkv, d]                   with cu_seqlens_k
 *        bf16 [num_pages, page_size, Hkv, d]      with block_table (paged)
 *   out  bf16, same shape as q (own strides)
 *   lse  fp32 [B, Hq, Sq], or [Hq, total_q] with cu_seqlens_q
 *   cu_seqlens_q / cu_seqlens_k  int32 [n_seq + 1] prefix sums of lengths
 *        (the flash_attn_varlen_func arguments of the same name); with a
 *        block_table, cu_seqlens_k gives each sequence's key count.
 *   block_table  int32 [n_seq, max_pages]: key j of sequence s is row
 *        j % page_size of page block_table[s][j / page_size].
 *   head dim d is 64 or 128.
 *
 * Ownership and synchronisation: every buffer belongs to the caller and lives
 * in device memory (except fa_tensor/fa_mask/fa_opts structs themselves, and
 * the host outputs of the query functions).  The library allocates no memory;
 * the caller passes a workspace of at least fa_fwd_workspace_size() bytes.
 * fa_fwd() only enqueues kernels on opts->stream and returns; it never
 * synchronises.  There is no CPU fallback and no alternative backend: on a
 * device that is not sm_103 the call fails with FA_ERR_NO_DEVICE.
 *
 * Errors: every entry point returns an fa_status.  Argument errors are found
 * on the host before anything is enqueued.  Faults found by kernels (a page
 * index outside the cache, a bounded wait that gave up) are recorded in an
 * error word in the first bytes of the workspace; fa_check_device_error()
 * reads and clears it.  The caller zero-fills the workspace's first 256 bytes
 * once, before its first use; fa_fwd never clears the word itself, so a fault
 * stays visible until it is checked.  The rest of those 256 bytes holds the
 * arrival counts of the prefill tail split (fa_plan.tail_units), which every
 * completed launch leaves at zero; fa_check_device_error clears all 256 bytes
 * when it finds a fault.  One workspace serves one call at a time.
 */
#ifndef MFA_GB300_FA_H
#define MFA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 8

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* bad dtype, shape, stride, alignment, Hq % Hkv, d, window, ... */
  FA_ERR_UNSUPPORTED = 2,    /* a valid combination the library does not implement */
  FA_ERR_WORKSPACE = 3,      /* workspace missing, too small or not 256-byte aligned */
  FA_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, tensor-map encode) */
  FA_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait gave up (reported by fa_check_device_error) */
  FA_ERR_DEVICE_BOUNDS = 6,  /* a kernel met an out-of-range index, e.g. a page (ditto) */
  FA_ERR_NO_DEVICE = 7,      /* no usable sm_103 device is current */
  FA_ERR_DEVICE_VALUE = 8    /* FA_DEBUG_VALIDATE found a mask value the call does not take (reported
                              * by fa_check_device_error; info = the mask tile or top-k bucket) */
} fa_status;

typedef enum { FA_DTYPE_BF16 = 1, FA_DTYPE_F32 = 2, FA_DTYPE_I32 = 3, FA_DTYPE_F16 = 4 } fa_dtype;

/* A strided view of device memory; shape/stride are in elements, outermost
 * first; only the first ndim entries are read. */
typedef struct {
  void* data;
  int32_t dtype; /* fa_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} fa_tensor;

typedef enum { FA_MASK_NONE = 0, FA_MASK_DENSE = 1, FA_MASK_TOPK = 2 } fa_mask_kind;

/* Additive mask.
 *  DENSE: t is fp32 [Sq, Sk] or [B|1, Hq|1, Sq, Sk]; a stride of 0 broadcasts.
 *         Entries must be finite or -inf.  Not combinable with cu_seqlens or
 *         block_table (FA_ERR_UNSUPPORTED).
 *  TOPK:  t is fp32 zero_hold_states [B, Hq, Sk]; keep_window >= 1.  Needs a
 *         fixed-length batch, Sk <= 16384, and no sliding window
 *         (FA_ERR_UNSUPPORTED otherwise). */
typedef struct {
  int32_t kind; /* fa_mask_kind */
  int32_t keep_window;
  fa_tensor t;
} fa_mask;

/* Debug flags (opts->debug_flags). */
#define FA_DEBUG_NO_SKIP 0x1u /* schedule EMPTY tiles too (as PARTIAL): exercises the -inf guard */
#define FA_DEBUG_WITHHOLD 0x2u /* test only: the prefill kernel's key producer withholds each CTA's first
                                * key tile (unmasked or dense-mask variants), so that the waits behind it
                                * give up after their bound (FA_ERR_DEVICE_TIMEOUT); the output is then
                                * undefined */
#define FA_DEBUG_VALIDATE 0x4u /* check mask values on the device: a dense mask must be finite or -inf,
                                * top-k scores finite (FA_ERR_DEVICE_VALUE otherwise); off by default */

typedef struct {
  void* stream;            /* cudaStream_t to enqueue on; NULL = legacy default stream */
  void* workspace;         /* device buffer, 256-byte aligned */
  size_t workspace_bytes;
  int32_t max_seqlen_q;    /* required with cu_seqlens_q: the longest query sequence */
  int32_t max_seqlen_k;    /* required with cu_seqlens_k: the longest key sequence */
  uint32_t debug_flags;
  int32_t reserved;
  /* Optional cudaEvent_t handles (NULL = none), recorded on `stream` right
   * before the main attention kernel is enqueued and right after its last
   * pass (split combine included): lets a caller time that kernel alone. */
  void* event_begin;
  void* event_end;
  /* Optional ALiBi slopes (NULL = none): device pointer to Hq fp32 values,
   * one per query head.  Adds -slope[h] * |i + kv_len - q_len - j| to the
   * (scaled, soft-capped) logit of query row i and key j, before masks:
   * vLLM pull request 11277, the `alibi_slopes` argument of its
   * flash_attn_varlen_func call (the pages give no formula; this linear
   * distance penalty, aligned bottom-right like the causal rule, is the plain
   * reading).  Read by the kernels, so it must stay valid until they finish.
 * On the prefill path ALiBi cannot be combined with a top-k mask
 * (FA_ERR_UNSUPPORTED); the decode path takes any combination. */
  const void* alibi_slopes;
  /* Optional cudaEvent_t (NULL = none), recorded on `stream` right after the
   * main attention kernel itself, before the split combine pass of the
   * decode path (for the prefill path, at the same point as event_end):
   * with event_begin it times the attention kernel alone.  fa_fwd and
   * fa_fwd_kvcache only. */
  void* event_attn_end;
} fa_opts;

/* Kernel path chosen by the planner. */
typedef enum { FA_PATH_DECODE = 1, FA_PATH_PREFILL = 2 } fa_path;

/* Tile classes produced by the scheduler. */
typedef enum { FA_TILE_EMPTY = 0, FA_TILE_FULL = 1, FA_TILE_PARTIAL = 2 } fa_tile_class;

/* The plan fa_fwd() would execute for given arguments (host-only query).
 *
 * Work is cut into items: item = (seq * n_heads_sched + head) * n_row_tiles
 * + row_tile.  For the PREFILL path head is a q-head and a row tile is
 * rows_per_tile query rows.  For the DECODE path head is a K/V head and a row
 * tile is 8 consecutive packed rows p = i * (Hq/Hkv) + (h % (Hq/Hkv)) of that
 * K/V head's query heads.  Keys are cut into tiles of keys_per_tile.
 *
 * Work list in the workspace after fa_fwd (device memory, int32), written by
 * the scheduler kernel on the DECODE path and on the PREFILL path with a
 * dense or top-k mask:
 *   counts[n_items]                   at workspace + off_counts
 *   tiles[n_items][n_k_tiles]         at workspace + off_tiles;
 *     entry = (k_tile << 1) | (class == FA_TILE_PARTIAL); only the first
 *     counts[item] entries are valid; EMPTY tiles never appear.
 * On the PREFILL path without a mask the pair rules alone classify the tiles,
 * so the attention kernel derives each item's list itself (the same tiles,
 * in the same order) and these two arrays are not written.
 *   stats: int64 [3] = tiles scheduled FULL, PARTIAL, and key tiles left out
 *     as EMPTY, at workspace + off_stats (every path).
 *   top-k masks only: int32 e[n_seq][Hq][Sk] at workspace + off_topk_e, the
 *     first query row at which key j is no longer kept (key j is kept on rows
 *     i with j <= i + Sk - Sq and i < e; INT32_MAX = never dropped,
 *     INT32_MIN = never kept).
 *   top-k masks on the PREFILL path: the keys some row of an item keeps,
 *     gathered (the attention kernel computes exactly these keys, as dense
 *     128-key tiles): counts[item] = number of gathered tiles and tiles[]
 *     entry t = (t << 1) | PARTIAL for gathered tile t (FULL: every row of
 *     the item keeps every key of the tile); at workspace + off_topk_list,
 *     per item n_k_tiles * 128 entries of two uint32, the first
 *     counts[item] * 128 set: first the keys every row of the item keeps,
 *     then the others, each group in key order; x = key | lo << 16 |
 *     hi << 24 where the item's rows row0 + lo .. row0 + hi - 1 keep the key
 *     (row0 = first row of the item; lo = 128, hi = 0 pads the last tile),
 *     y = the key's bias z * log2(e) as fp32 bits. */
typedef struct {
  int32_t path;            /* fa_path */
  int32_t n_seq;
  int32_t n_heads_sched;
  int32_t n_row_tiles;
  int32_t rows_per_tile;   /* query rows (PREFILL) or packed rows (DECODE) per item */
  int32_t keys_per_tile;
  int32_t n_k_tiles;       /* key tiles of the longest key sequence */
  int32_t n_splits;        /* DECODE: key splits per item (1 = no combine pass) */
  int32_t tiles_per_split; /* DECODE: key tiles per split */
  int32_t tail_units;      /* PREFILL: units of the persistent grid's last round
                              that two CTAs run as halves of their key tiles and
                              merge by LSE (0 = none) */
  int64_t n_items;
  size_t off_counts;
  size_t off_tiles;
  size_t off_stats;
  size_t off_topk_e;       /* 0 unless the mask is FA_MASK_TOPK */
  size_t off_topk_list;    /* 0 unless FA_MASK_TOPK on the PREFILL path */
  int64_t n_kernels;       /* kernel launches one fa_fwd call enqueues */
  size_t workspace_bytes;  /* minimum workspace size */
} fa_plan;

/* Masked attention forward; see the file comment for the semantics.
 *   scale <= 0 selects 1/sqrt(d); softcap == 0 disables the soft-cap;
 *   window_left / window_right == -1 leave that side unbounded; causal != 0
 *   applies the bottom-right causal rule. */
int fa_fwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
           const fa_tensor* out, const fa_tensor* lse,
           const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
           const fa_tensor* block_table, const fa_mask* mask,
           int32_t window_left, int32_t window_right, float softcap, float scale,
           int32_t causal, const fa_opts* opts);

/* Debug dump: fa_fwd (no page table, no mask, bf16, prefill path, no ALiBi;
 * FA_ERR_UNSUPPORTED otherwise) through a debug build of the prefill kernel
 * that also copies, for the 128 query rows of tile `row_tile` of sequence
 * `seq` and q-head `head`, the intermediate values of every key tile that
 * unit visits, into the caller's device buffer `dump` (fp32):
 *   S[it][row][key]          raw Q K^T, before scale and masks, at dump;
 *   P[it][row][key]          the probabilities as rounded for P V (0 where a
 *                            key is dropped), at dump + n_k_tiles * 128 * 128;
 *   ref[it][row]             the row's exponent reference in log2 units
 *                            (P = exp2(logit * log2 e - ref)), at
 *                            dump + 2 * n_k_tiles * 128 * 128.
 * Entry it is the it-th key tile of the unit's list; the debug build writes
 * that unit's count and list into the workspace work list (counts[item],
 * tiles[item][...], as documented for fa_fwd_plan) whichever path scheduled
 * it.  dump_bytes must be at least fa_debug_dump_bytes(n_k_tiles of the
 * plan); entries past the list's end are left unwritten.  The output and LSE
 * are as fa_fwd's.  A dump of one block's intermediate values for
 * step-by-step comparison, as flash-sparse-attention issue 11 "Next Steps"
 * proposes for its minimal example. */
int fa_fwd_debug_dump(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                      const fa_tensor* lse, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                      int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
                      const fa_opts* opts, int32_t seq, int32_t head, int32_t row_tile, float* dump,
                      size_t dump_bytes);
size_t fa_debug_dump_bytes(int64_t n_k_tiles);

/* Host-only: validate the arguments of fa_fwd and describe its plan
 * (pointers are checked for alignment but never dereferenced; opts->workspace
 * may be NULL).  Same status codes as fa_fwd, except FA_ERR_WORKSPACE. */
int fa_fwd_plan(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                const fa_tensor* out, const fa_tensor* lse,
                const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                const fa_tensor* block_table, const fa_mask* mask,
                int32_t window_left, int32_t window_right, float softcap, float scale,
                int32_t causal, const fa_opts* opts, fa_plan* plan_out);

/* Host-only: minimum workspace size for these arguments (fa_fwd_plan's
 * workspace_bytes). */
int fa_fwd_workspace_size(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                          const fa_tensor* out, const fa_tensor* lse,
                          const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                          const fa_tensor* block_table, const fa_mask* mask,
                          int32_t window_left, int32_t window_right, float softcap,
                          float scale, int32_t causal, const fa_opts* opts, size_t* bytes);

/* Attention over a KV cache plus the step's active keys, read from two
 * sources (vLLM pull request 11277, the author's reply on aligning with the
 * unified flash_attn_varlen_func interface, first point: writing the new
 * tokens into the cache before the attention reads them back is a
 * read-after-write stall, so the cached and the active K/V are passed
 * separately).  Sequence s has keys, in order, cache rows 0 .. L_s - 1
 * (L_s = cache_seqlens[s]) followed by its active rows 0 .. q_len_s - 1, the
 * keys of its own query tokens: kv_len_s = L_s + q_len_s, and the causal rule
 * (bottom-right) lets query row i see cached keys and active keys 0 .. i.
 * The active rows are read from k_new / v_new, never from the cache.
 *
 *   q             as for fa_fwd: [B, Sq, Hq, d], or [total_q, Hq, d] with
 *                 cu_seqlens_q
 *   k_new, v_new  the active keys/values, laid out like q with Hkv heads:
 *                 [B, Sq, Hkv, d] or [total_q, Hkv, d]
 *   k_cache, v_cache  paged [num_pages, page_size, Hkv, d] with block_table
 *                 [n_seq, max_pages] (cache row j of sequence s is row
 *                 j % page_size of page block_table[s][j / page_size]), or
 *                 padded [n_seq, cap, Hkv, d] without a block table
 *   cache_seqlens int32 [n_seq], device: keys already in the cache
 *   append != 0   also write the active rows into the cache at rows
 *                 L_s .. L_s + q_len_s - 1 (a bit-exact copy, done by the
 *                 attention kernel itself from the active tensors; no kernel
 *                 of this call reads those cache rows)
 *   out, lse      as for fa_fwd
 * The element type rule, GQA, window, softcap, scale, ALiBi (opts) and the
 * fully-masked-row rule are those of fa_fwd; dense and top-k masks return
 * FA_ERR_UNSUPPORTED.  opts->max_seqlen_k is required: the largest
 * L_s + q_len_s.  Work runs on the split-KV decode kernel whatever q_len is.
 * A cached or appended row beyond the cache (block table width x page_size,
 * or cap) or a bad page index is recorded as FA_ERR_DEVICE_BOUNDS and its
 * access skipped; a sequence with L_s + q_len_s > max_seqlen_k is rejected
 * the same way as in fa_fwd. */
int fa_fwd_kvcache(const fa_tensor* q, const fa_tensor* k_cache, const fa_tensor* v_cache,
                   const fa_tensor* k_new, const fa_tensor* v_new, const fa_tensor* out,
                   const fa_tensor* lse, const fa_tensor* cu_seqlens_q,
                   const fa_tensor* cache_seqlens, const fa_tensor* block_table,
                   int32_t window_left, int32_t window_right, float softcap, float scale,
                   int32_t causal, int32_t append, const fa_opts* opts);

/* Host-only: validate the arguments of fa_fwd_kvcache and describe its plan
 * (as fa_fwd_plan). */
int fa_fwd_kvcache_plan(const fa_tensor* q, const fa_tensor* k_cache, const fa_tensor* v_cache,
                        const fa_tensor* k_new, const fa_tensor* v_new, const fa_tensor* out,
                        const fa_tensor* lse, const fa_tensor* cu_seqlens_q,
                        const fa_tensor* cache_seqlens, const fa_tensor* block_table,
                        int32_t window_left, int32_t window_right, float softcap, float scale,
                        int32_t causal, int32_t append, const fa_opts* opts, fa_plan* plan_out);

/* Backward pass: dq, dk, dv of the forward for the same arguments
 * (InfiniTrain pull request 193, "FlashAttention native backend": the
 * FlashAttention-2 causal forward and backward kernels it builds; "Framework
 * 与 autograd": the autograd function around them).  With P recomputed from
 * the forward's LSE, Delta = rowsum(dout * out), dP = dout V^T and
 * dS = P * (dP - Delta) * dx/ds (dx/ds = scale, or scale * (1 - tanh^2) under
 * the soft-cap): dv = sum over a group's q-heads of P^T dout, dk = sum of
 * dS^T q, dq = dS k.  ALiBi (opts->alibi_slopes) enters the logits as in the
 * forward and gets no gradient.
 *   q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, window, softcap, scale,
 *                causal, opts: as given to fa_fwd (out and lse from it)
 *   dout, dq     laid out like q (own strides), the input element type
 *   dk, dv       laid out like k (own strides), the input element type
 * No paged cache and no dense or top-k mask (the call takes neither).  The
 * result does not depend on scheduling: no atomics, every gradient row is
 * summed in a fixed order by one CTA.  dq/dk/dv rows of keys or queries
 * that no pair reaches are written as 0.  Workspace: fa_bwd_plan's
 * workspace_bytes (the forward's plus Delta, fp32 per query row and head). */
int fa_bwd(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
           const fa_tensor* lse, const fa_tensor* dout, const fa_tensor* dq, const fa_tensor* dk,
           const fa_tensor* dv, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
           int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
           const fa_opts* opts);

/* Host-only: validate the arguments of fa_bwd and describe its plan (as
 * fa_fwd_plan; n_kernels counts the Delta, dk/dv and dq kernels). */
int fa_bwd_plan(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, const fa_tensor* out,
                const fa_tensor* lse, const fa_tensor* dout, const fa_tensor* dq, const fa_tensor* dk,
                const fa_tensor* dv, const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                int32_t window_left, int32_t window_right, float softcap, float scale, int32_t causal,
                const fa_opts* opts, fa_plan* plan_out);

/* Size of the static device scratch used by fa_fwd_noalloc (32 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* fa_fwd for callers that cannot allocate device memory (the pages this
 * library follows have no counterpart of it).  Some callers may not call
 * cudaMalloc at all: allocator-free inference runtimes that only hand out
 * pre-sized input/output buffers, plugins whose host forbids device
 * allocations after start-up, latency paths that must not touch an allocator.
 * This entry point takes the same arguments as fa_fwd, except that
 * opts->workspace and opts->workspace_bytes are ignored: the scratch lives in
 * a static device array of FA_NOALLOC_SCRATCH_BYTES that the library owns and
 * that every GPU loading the library holds until the process exits.  It calls
 * no allocating routine.
 *   - A problem whose scratch need (fa_fwd_workspace_size) exceeds
 *     FA_NOALLOC_SCRATCH_BYTES is rejected with FA_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (a
 *     one-time set-up per device, done with that device current, and done
 *     again only if the device's context was destroyed and re-created, e.g.
 *     after cudaDeviceReset); make that first call before any stream capture.
 *   - All calls share the array: calls that overlap on the GPU (other
 *     streams, other threads) race on it; serialise them.
 *   - Each call clears the array's device error word before its kernels run,
 *     and the word cannot be read back, so nothing the kernels record there
 *     reaches the caller: a bad page index or inconsistent sequence lengths
 *     (FA_ERR_DEVICE_BOUNDS) and a bounded wait that gave up
 *     (FA_ERR_DEVICE_TIMEOUT) still return FA_OK, with `out` not valid.  Use
 *     fa_fwd with a workspace and fa_check_device_error when that matters.
 *   - For the same reason opts->debug_flags with FA_DEBUG_VALIDATE (whose
 *     only result is FA_ERR_DEVICE_VALUE in that word) is refused with
 *     FA_ERR_UNSUPPORTED. */
int fa_fwd_noalloc(const fa_tensor* q, const fa_tensor* k, const fa_tensor* v,
                   const fa_tensor* out, const fa_tensor* lse,
                   const fa_tensor* cu_seqlens_q, const fa_tensor* cu_seqlens_k,
                   const fa_tensor* block_table, const fa_mask* mask,
                   int32_t window_left, int32_t window_right, float softcap, float scale,
                   int32_t causal, const fa_opts* opts);

/* Synchronises `stream`, then reads and clears the device error word at the
 * start of `workspace`: FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_DEVICE_BOUNDS.
 * `info` (nullable) receives the first recorded detail (e.g. the bad page). */
int fa_check_device_error(void* stream, void* workspace, uint32_t* info);

/* Static text for a status code. */
const char* fa_status_string(int status);

/* FA_ABI_VERSION of the loaded library. */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MFA_GB300_FA_H */
