"""Keys from two sources, and the cache append -- test infrastructure.

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of the
benchmark may use this module; the CUDA library never does.

vLLM pull request 11277, the author's reply on aligning with the unified
``flash_attn_varlen_func`` interface, first point: instead of writing the
step's new tokens into the KV cache (``reshape_and_cache_flash``) and reading
them back, the cached K/V and the active K/V are passed to the attention
separately.  The plain reading taken here: sequence s sees, in order, its
``cache_seqlens[s]`` cached keys and then the keys of its own query tokens
(one active row per query row), so ``kv_len = cache_seqlens[s] + q_len`` and
the bottom-right causal rule lets query row i see every cached key and active
keys 0..i.  The optional append writes the active rows into the cache right
after the cached ones, unchanged.
"""
from __future__ import annotations

import numpy as np

from .attention import _np, attention, gather_paged


def cached_rows(cache, b, n, block_table=None):
    """The first ``n`` cached rows ``[n, H, d]`` of sequence ``b``: from a paged
    cache ``[num_pages, page_size, H, d]`` through ``block_table`` (page
    ``block_table[b][j // page_size]``, row ``j % page_size``), or from a
    padded cache ``[n_seq, cap, H, d]``."""
    cache = _np(cache)
    if block_table is not None:
        return gather_paged(cache, _np(block_table, np.int64)[b], n)
    return cache[b, :n]


def active_rows(x, b, cu_seqlens_q=None):
    """Sequence ``b``'s active rows: ``x[cu[b]:cu[b+1]]`` when packed, else
    ``x[b]``."""
    x = _np(x)
    if cu_seqlens_q is not None:
        cu = _np(cu_seqlens_q, np.int64)
        return x[int(cu[b]):int(cu[b + 1])]
    return x[b]


def full_keys(k_cache, v_cache, k_new, v_new, cache_seqlens, cu_seqlens_q=None, block_table=None):
    """Packed ``[total_k, Hkv, d]`` keys and values (cached rows, then active
    rows, per sequence) and their ``cu_seqlens_k``."""
    lens = _np(cache_seqlens, np.int64)
    ks, vs, cu = [], [], [0]
    for b in range(len(lens)):
        kc = cached_rows(k_cache, b, int(lens[b]), block_table)
        vc = cached_rows(v_cache, b, int(lens[b]), block_table)
        ka = active_rows(k_new, b, cu_seqlens_q)
        va = active_rows(v_new, b, cu_seqlens_q)
        ks.append(np.concatenate([kc, ka], axis=0))
        vs.append(np.concatenate([vc, va], axis=0))
        cu.append(cu[-1] + ks[-1].shape[0])
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0), np.asarray(cu, dtype=np.int64)


def attention_kvcache(q, k_cache, v_cache, k_new, v_new, cache_seqlens, *, cu_seqlens_q=None,
                      block_table=None, **kw):
    """Attention of ``q`` over each sequence's cached keys followed by its
    active keys; the remaining keyword arguments (scale, causal, window,
    softcap, alibi_slopes) are those of ``attention``.  Returns ``(out, lse)``
    as ``attention`` does for this ``q`` layout."""
    K, V, cu_k = full_keys(k_cache, v_cache, k_new, v_new, cache_seqlens, cu_seqlens_q, block_table)
    return attention(q, K, V, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_k, **kw)


def append_kvcache(k_cache, v_cache, k_new, v_new, cache_seqlens, *, cu_seqlens_q=None, block_table=None):
    """The caches after the append: copies in which the active rows of
    sequence b occupy cache rows ``cache_seqlens[b] .. + q_len - 1``."""
    kc = np.array(_np(k_cache), copy=True)
    vc = np.array(_np(v_cache), copy=True)
    lens = _np(cache_seqlens, np.int64)
    bt = None if block_table is None else _np(block_table, np.int64)
    for b in range(len(lens)):
        ka = active_rows(k_new, b, cu_seqlens_q)
        va = active_rows(v_new, b, cu_seqlens_q)
        for t in range(ka.shape[0]):
            j = int(lens[b]) + t
            if bt is not None:
                page, row = int(bt[b][j // kc.shape[1]]), j % kc.shape[1]
                kc[page, row] = ka[t]
                vc[page, row] = va[t]
            else:
                kc[b, j] = ka[t]
                vc[b, j] = va[t]
    return kc, vc
