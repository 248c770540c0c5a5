"""Seeded synthetic inputs for masked flash-attention (forward).

This module only draws inputs: random Q/K/V, masks, top-k scores, sequence
lengths, page tables.  It holds none of the attention arithmetic, so both the
CPU oracle and the CUDA path can be fed from it without sharing any of the
method.  Every tensor is a CPU torch tensor; callers move them where needed.

Recipe (shared by tests and the benchmark):
  * one ``torch.Generator`` seeded with ``seed``; tensors are drawn in the
    order they are listed in each builder;
  * Q/K/V are fp32 N(0,1) rounded to bf16, layout ``[batch, seq, heads, d]``
    (``bshd``), or ``[total, heads, d]`` for packed variable-length batches;
  * top-k scores ``zero_hold_states`` are fp32 N(0,1), ``[batch, heads, keys]``;
  * paged K/V caches are ``[num_pages, page_size, heads, d]`` and the page
    table is a random permutation of the pages, ``-1`` past a sequence's end.

The named workloads follow the shapes the flash-attention pages discuss: the
ExecuTorch sliding-window decode example (700-key cache, keys 515..575 kept),
causal prefill over past KV with grouped-query heads (FastChat, InfiniTrain),
GPT-2 / Llama-3 training-layer shapes (InfiniTrain), a vLLM-style varlen paged
decode batch with window and softcap, and flash-sparse-attention's dynamic
top-k mask.
"""
from __future__ import annotations

import math

import torch

BF16 = torch.bfloat16


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def randn_bf16(g: torch.Generator, shape, dtype=BF16) -> torch.Tensor:
    """fp32 N(0, 1) draws rounded to the input type (bf16, or fp16)."""
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def qkv_bshd(g, B, Sq, Sk, Hq, Hkv, d, dtype=BF16):
    q = randn_bf16(g, (B, Sq, Hq, d), dtype)
    k = randn_bf16(g, (B, Sk, Hkv, d), dtype)
    v = randn_bf16(g, (B, Sk, Hkv, d), dtype)
    return q, k, v


def base_params(**kw):
    p = dict(scale=None, causal=False, window_left=-1, window_right=-1,
             softcap=0.0, mask=None, zero_hold_states=None, keep_window=0,
             cu_seqlens_q=None, cu_seqlens_k=None, block_table=None,
             max_seqlen_q=None, max_seqlen_k=None)
    p.update(kw)
    return p


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------

def sliding_window_decode(seed: int = 0, all_masked: bool = False):
    """700-key cache, one query at position 575, additive mask that keeps keys
    515..575 (the query and the 60 before it) and is -inf everywhere else; the
    first 512-key chunk is therefore entirely -inf.  ``all_masked`` makes the
    whole row -inf (the row must come out as O=0, LSE=-inf).
    B=1, Hq=Hkv=1, d=64, not causal (the mask alone selects the keys)."""
    g = _gen(seed)
    q, k, v = qkv_bshd(g, 1, 1, 700, 1, 1, 64)
    mask = torch.full((1, 700), float("-inf"), dtype=torch.float32)
    if not all_masked:
        mask[0, 515:576] = 0.0
    return dict(name="sliding_window_decode_kv700", q=q, k=k, v=v,
                params=base_params(scale=1.0 / 8.0, mask=mask))


def causal_prefill_past_kv(seed: int = 0, B=4, Hq=32, Hkv=8, d=128, q_len=512, kv_len=4096):
    """Causal prefill of ``q_len`` new tokens over ``kv_len - q_len`` cached
    ones (bottom-right aligned causal mask), grouped-query heads."""
    g = _gen(seed)
    q, k, v = qkv_bshd(g, B, q_len, kv_len, Hq, Hkv, d)
    return dict(name=f"causal_prefill_gqa_b{B}_hq{Hq}_hkv{Hkv}_d{d}_q{q_len}_kv{kv_len}",
                q=q, k=k, v=v, params=base_params(scale=1.0 / math.sqrt(d), causal=True))


def causal_self_attention(seed: int = 0, B=8, T=1024, Hq=12, Hkv=12, d=64):
    """Square causal self-attention at training-layer shapes: GPT-2 small
    (B=8, T=1024, 12 heads, d=64) or Llama-3-8B (B=1, T=8192, 32/8 heads,
    d=128)."""
    g = _gen(seed)
    q, k, v = qkv_bshd(g, B, T, T, Hq, Hkv, d)
    return dict(name=f"causal_self_b{B}_t{T}_hq{Hq}_hkv{Hkv}_d{d}", q=q, k=k, v=v,
                params=base_params(scale=1.0 / math.sqrt(d), causal=True))


def gpt2_small_layer(seed: int = 0):
    return causal_self_attention(seed, B=8, T=1024, Hq=12, Hkv=12, d=64)


def llama3_8b_layer(seed: int = 0):
    return causal_self_attention(seed, B=1, T=8192, Hq=32, Hkv=8, d=128)


def paged_varlen_decode(seed: int = 0, n_seq=64, min_len=128, max_len=8192, Hq=32, Hkv=8,
                        d=128, page_size=16, window_left=4096, softcap=30.0):
    """Batch of ``n_seq`` single-token decodes over a paged KV cache.  Key
    lengths are uniform in [min_len, max_len]; the page table is a random
    permutation of all pages.  Sliding window ``window_left`` keys to the left,
    causal, logit softcap."""
    g = _gen(seed)
    lens = torch.randint(min_len, max_len + 1, (n_seq,), generator=g, dtype=torch.int64)
    pages_per = [(int(L) + page_size - 1) // page_size for L in lens]
    n_pages = sum(pages_per)
    max_pages = max(pages_per)
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    block_table = torch.full((n_seq, max_pages), -1, dtype=torch.int32)
    pos = 0
    for s, n in enumerate(pages_per):
        block_table[s, :n] = perm[pos:pos + n]
        pos += n
    q = randn_bf16(g, (n_seq, Hq, d))
    k_cache = randn_bf16(g, (n_pages, page_size, Hkv, d))
    v_cache = randn_bf16(g, (n_pages, page_size, Hkv, d))
    cu_q = torch.arange(0, n_seq + 1, dtype=torch.int32)
    cu_k = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_k[1:] = torch.cumsum(lens, 0).to(torch.int32)
    return dict(name=f"paged_varlen_decode_n{n_seq}_hq{Hq}_hkv{Hkv}_d{d}_page{page_size}",
                q=q, k=k_cache, v=v_cache, kv_lens=lens.to(torch.int32),
                params=base_params(scale=1.0 / math.sqrt(d), causal=True,
                                   window_left=window_left, window_right=0, softcap=softcap,
                                   cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                                   block_table=block_table, max_seqlen_q=1,
                                   max_seqlen_k=int(lens.max())))


def paged_decode_append(seed: int = 0, **kw):
    """The paged varlen decode batch served the two-source way: each
    sequence's newest token is the active row (``k_new``/``v_new``), the
    ``kv_len - 1`` before it are cached, and the call appends the active row
    to the cache.  The cache already holds that row's values, so the keys the
    attention sees, and the cache after the append, equal the paged workload's."""
    c = paged_varlen_decode(seed, **kw)
    lens = c["kv_lens"].to(torch.int64)
    bt = c["params"]["block_table"]
    page = c["k"].shape[1]
    last = lens - 1
    pages = bt[torch.arange(len(lens)), last // page].to(torch.int64)
    rows = last % page
    k_new = c["k"][pages, rows]      # [n_seq, Hkv, d]: one active row per sequence
    v_new = c["v"][pages, rows]
    c = dict(c, name=c["name"].replace("paged_varlen_decode", "paged_decode_append"))
    c["kvcache"] = dict(k_new=k_new, v_new=v_new, cache_seqlens=last.to(torch.int32), append=True)
    return c


def dynamic_topk(seed: int = 0, B=2, H=16, d=128, T=8192, keep_window=2048):
    """Causal attention where each query row keeps only the ``keep_window``
    causally-allowed keys with the largest ``zero_hold_states`` value; the kept
    keys get that value added to their logit."""
    g = _gen(seed)
    q, k, v = qkv_bshd(g, B, T, T, H, H, d)
    z = torch.randn(B, H, T, generator=g, dtype=torch.float32)
    return dict(name=f"dynamic_topk_b{B}_h{H}_d{d}_t{T}_keep{keep_window}", q=q, k=k, v=v,
                params=base_params(scale=1.0 / math.sqrt(d), causal=True,
                                   zero_hold_states=z, keep_window=keep_window))


# ---------------------------------------------------------------------------
# Small random cases (parity sweeps)
# ---------------------------------------------------------------------------

def random_case(seed, B=1, Sq=1, Sk=1, Hq=1, Hkv=1, d=64, dtype=BF16, **params):
    g = _gen(seed)
    q, k, v = qkv_bshd(g, B, Sq, Sk, Hq, Hkv, d, dtype)
    p = base_params(scale=1.0 / math.sqrt(d))
    p.update(params)
    return dict(name=f"rand_s{seed}_b{B}_q{Sq}_k{Sk}_h{Hq}x{Hkv}_d{d}", q=q, k=k, v=v, params=p)


def random_dense_mask(seed, Sq, Sk, p_neg_inf=0.3, p_zero=0.3):
    """fp32 additive mask with a mix of -inf, 0 and N(0,1) biases."""
    g = _gen(seed + 7919)
    u = torch.rand(Sq, Sk, generator=g)
    vals = torch.randn(Sq, Sk, generator=g)
    m = torch.where(u < p_neg_inf, torch.full_like(vals, float("-inf")),
                    torch.where(u < p_neg_inf + p_zero, torch.zeros_like(vals), vals))
    return m.to(torch.float32)


def random_zero_hold_states(seed, B, H, Sk, ties=False):
    g = _gen(seed + 104729)
    z = torch.randn(B, H, Sk, generator=g, dtype=torch.float32)
    if ties:  # quantise so equal values (ties) are common
        z = torch.round(z * 2.0) / 2.0
    return z


def random_varlen(seed, n_seq, max_q, max_k, Hq, Hkv, d, q_eq_k=False, min_q=0, min_k=0, dtype=BF16):
    """Packed variable-length batch: per-sequence lengths drawn uniformly."""
    g = _gen(seed)
    lq = torch.randint(min_q, max_q + 1, (n_seq,), generator=g)
    if q_eq_k:
        lk = lq.clone()
    else:
        lk = torch.randint(min_k, max_k + 1, (n_seq,), generator=g)
    cu_q = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_k = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(lq, 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(lk, 0).to(torch.int32)
    q = randn_bf16(g, (int(cu_q[-1]), Hq, d), dtype)
    k = randn_bf16(g, (int(cu_k[-1]), Hkv, d), dtype)
    v = randn_bf16(g, (int(cu_k[-1]), Hkv, d), dtype)
    return q, k, v, cu_q, cu_k


def paginate(k, v, cu_k, page_size, seed):
    """Scatter a packed [total, H, d] K/V into a paged cache with a random
    permutation of pages; returns (k_cache, v_cache, block_table)."""
    g = _gen(seed + 15485863)
    n_seq = cu_k.numel() - 1
    lens = [int(cu_k[s + 1] - cu_k[s]) for s in range(n_seq)]
    pages_per = [(L + page_size - 1) // page_size for L in lens]
    n_pages = max(1, sum(pages_per))
    H, d = k.shape[1], k.shape[2]
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    kc = torch.zeros(n_pages, page_size, H, d, dtype=k.dtype)
    vc = torch.zeros(n_pages, page_size, H, d, dtype=v.dtype)
    bt = torch.full((n_seq, max(1, max(pages_per) if pages_per else 1)), -1, dtype=torch.int32)
    pos = 0
    for s in range(n_seq):
        base = int(cu_k[s])
        for p in range(pages_per[s]):
            page = int(perm[pos])
            pos += 1
            bt[s, p] = page
            lo = p * page_size
            hi = min(lens[s], lo + page_size)
            kc[page, :hi - lo] = k[base + lo: base + hi]
            vc[page, :hi - lo] = v[base + lo: base + hi]
    return kc, vc, bt


WORKLOADS = {
    "paged_decode_append": paged_decode_append,
    "sliding_window_decode": sliding_window_decode,
    "causal_prefill_past_kv": causal_prefill_past_kv,
    "gpt2_small_layer": gpt2_small_layer,
    "llama3_8b_layer": llama3_8b_layer,
    "paged_varlen_decode": paged_varlen_decode,
    "dynamic_topk": dynamic_topk,
}
