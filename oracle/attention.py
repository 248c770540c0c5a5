"""fp64 numpy definition of masked attention (forward) -- test infrastructure.

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of the
benchmark may use this module; the CUDA library never does.

What is computed (for every sequence b, query head h, query row i, key j):

  1. grouped-query heads: K/V head ``g = h // (Hq // Hkv)``; the rule that Hq
     must be a multiple of Hkv, with MHA when equal and GQA/MQA otherwise, is
     InfiniTrain pull request 193 "feat: Flash Attention", section
     "Framework 与 autograd"; sharing the original K/V heads instead of
     repeating them is its section "Transformer 接入".
  2. ``x = scale * <Q[i], K[j]>``, then the logit soft-cap
     ``x = softcap * tanh(x / softcap)`` when softcap > 0 (the ``softcap``
     argument of the vLLM pull request 11277 ``flash_attn_varlen_func`` call),
     then the ALiBi bias ``x -= slope[h] * |i + off - j|`` when per-head slopes
     are given (the ``alibi_slopes`` argument of the same call; the pages name
     it without a formula, and this linear distance penalty, aligned like the
     causal rule below, is its plain reading).
  3. pair rules, with ``off = kv_len - q_len`` (bottom-right alignment: the
     last query sits on the last key; FastChat pull request 2315 "Optimize
     for proper flash attn causal handling", causal with q_len != kv_len and
     past key-values without padding q):
       causal        -> j <= i + off
       window_left   -> j >= i + off - window_left   (when >= 0)
       window_right  -> j <= i + off + window_right  (when >= 0)
       length        -> 0 <= j < kv_len
  4. additive terms, added after the soft-cap: a dense mask ``M[i, j]``
     (ExecuTorch pull request 10466, "Summary": a [q_len, kv_len] mask added
     to q@k, -inf to drop a key), or the dynamic top-k mask of
     flash-sparse-attention issue 11 "[Integration Progress Report] Dynamic
     Mask Attention Integration into FlashAttention" ("Overview" part 1 and
     "Next Steps" 1): among the keys that rule 3 allows for row i, the
     ``keep_window`` with the largest ``zero_hold_states[b, h, j]`` are kept
     (ties: the lower key index wins) and get that value added to their
     logit; every other key is -inf.
  5. a row whose logits are all -inf (ExecuTorch "Summary": a fully -inf
     chunk) gives O = 0 and LSE = -inf; otherwise the plain softmax
     ``p = exp(x - max) / sum``, ``O = p @ V``, ``LSE = max + ln(sum)``.

Where the pages are silent the plainest reading that the rest supports is
taken; each such reading is stated where it is used.
"""
from __future__ import annotations

import numpy as np


def _np(a, dtype=np.float64):
    """Convert a numpy array or CPU torch tensor to numpy of ``dtype``."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        t = a.detach()
        if t.dtype.is_floating_point:
            t = t.double()  # exact for bf16, fp16, fp32 and fp64 inputs
        a = t.cpu().numpy()
    return np.asarray(a, dtype=dtype)


def allowed_pairs(rows, keys, q_len, kv_len, causal=False, window_left=-1, window_right=-1):
    """Boolean ``[len(rows), len(keys)]``: pairs kept by the causal (bottom-right),
    sliding-window and length rules (rule 3 of the module docstring)."""
    off = int(kv_len) - int(q_len)
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(keys, dtype=np.int64)[None, :]
    ok = (j >= 0) & (j < kv_len) & (i >= 0) & (i < q_len)
    if causal:
        ok = ok & (j <= i + off)
    if window_left is not None and window_left >= 0:
        ok = ok & (j >= i + off - window_left)
    if window_right is not None and window_right >= 0:
        ok = ok & (j <= i + off + window_right)
    return ok


def topk_kept_row(z, candidates, keep_window):
    """Indices of the kept keys for one query row of the dynamic top-k mask.

    ``candidates`` is a boolean vector of keys allowed by the pair rules; the
    ``keep_window`` candidates with the largest ``z`` are kept, ties going to
    the lower key index; with fewer candidates than ``keep_window`` all are
    kept.  A plain sort of the candidates (flash-sparse-attention issue 11,
    "Overview": causal masking and top-k selection)."""
    idx = np.nonzero(np.asarray(candidates))[0]
    if len(idx) <= keep_window:
        return idx
    zc = np.asarray(z, dtype=np.float64)[idx]
    order = np.lexsort((idx, -zc))  # primary: z descending, secondary: index ascending
    return np.sort(idx[order[:keep_window]])


def logits_rows(q_rows, k, rows, q_len, kv_len, *, scale, causal=False, window_left=-1,
                window_right=-1, softcap=0.0, mask_rows=None, z=None, keep_window=0,
                alibi_slope=None):
    """Final logits ``x[r, j]`` for the query rows ``rows`` of one (sequence,
    head): scaled dot products, soft-cap, pair rules, additive terms; -inf
    where a key is dropped.  ``q_rows`` is ``[len(rows), d]``, ``k`` is
    ``[kv_len, d]``, ``mask_rows`` is ``[len(rows), kv_len]``, ``z`` is
    ``[kv_len]``."""
    q_rows = _np(q_rows)
    k = _np(k)
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.arange(kv_len)
    s = float(scale) * (q_rows @ k.T)
    if softcap and softcap > 0:
        s = float(softcap) * np.tanh(s / float(softcap))
    if alibi_slope is not None:  # this head's ALiBi slope
        off = kv_len - q_len
        s = s - float(alibi_slope) * np.abs((rows + off)[:, None] - keys[None, :]).astype(np.float64)
    ok = allowed_pairs(rows, keys, q_len, kv_len, causal, window_left, window_right)
    if mask_rows is not None:
        s = s + _np(mask_rows)
    if z is not None:
        z = _np(z)
        keep = np.zeros_like(ok)
        for r in range(len(rows)):
            keep[r, topk_kept_row(z, ok[r], keep_window)] = True
        ok = keep
        s = s + z[None, :]
    return np.where(ok, s, -np.inf)


def softmax_rows(x):
    """Row softmax of logits with -inf entries.  Returns ``(p, lse)``; a row
    with no finite logit gives p = 0 and lse = -inf (never NaN)."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[1] == 0:
        return np.zeros_like(x), np.full(x.shape[0], -np.inf)
    m = x.max(axis=1)
    empty = ~(m > -np.inf)
    m_ref = np.where(empty, 0.0, m)
    e = np.exp(x - m_ref[:, None])
    ssum = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, ssum)[:, None])
        lse = np.where(empty, -np.inf, m_ref + np.log(np.where(empty, 1.0, ssum)))
    return p, lse


def attention_rows(q_rows, k, v, rows, q_len, kv_len, **kw):
    """Output and LSE for selected query rows of one (sequence, head)."""
    x = logits_rows(q_rows, k, rows, q_len, kv_len, **kw)
    p, lse = softmax_rows(x)
    return p @ _np(v), lse


def gather_paged(cache, block_table_row, kv_len):
    """Logical ``[kv_len, H, d]`` keys (or values) of one sequence from a paged
    cache ``[num_pages, page_size, H, d]`` (the vLLM ``block_table``
    argument): key j lives at page ``block_table_row[j // page_size]``, row
    ``j % page_size``."""
    cache = np.asarray(cache)
    page_size = cache.shape[1]
    j = np.arange(kv_len)
    pages = np.asarray(block_table_row, dtype=np.int64)[j // page_size]
    return cache[pages, j % page_size]


def _mask_for(mask, b, h, Sq, Sk):
    if mask is None:
        return None
    m = _np(mask)
    if m.ndim == 2:
        return np.broadcast_to(m, (Sq, Sk))
    if m.ndim == 4:
        return np.broadcast_to(m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0], (Sq, Sk))
    raise ValueError("mask must be [q_len, kv_len] or [B|1, H|1, q_len, kv_len]")


def attention(q, k, v, *, scale=None, causal=False, window_left=-1, window_right=-1,
              softcap=0.0, mask=None, zero_hold_states=None, keep_window=0,
              cu_seqlens_q=None, cu_seqlens_k=None, block_table=None, alibi_slopes=None,
              **_unused):
    """Masked attention forward over a whole batch.

    Layouts: Q ``[B, Sq, Hq, d]`` and K/V ``[B, Sk, Hkv, d]``; or packed
    variable-length Q ``[total_q, Hq, d]`` with ``cu_seqlens_q`` and K/V
    ``[total_k, Hkv, d]`` with ``cu_seqlens_k`` (vLLM ``flash_attn_varlen_func``
    arguments); or a paged K/V cache ``[num_pages, page_size, Hkv, d]`` with
    ``block_table`` ``[n_seq, max_pages]`` and ``cu_seqlens_k`` giving each
    sequence's key count; ``alibi_slopes``, optional, per q-head ``[Hq]``.
    Returns ``(out, lse)`` in fp64: ``out`` shaped like
    Q; ``lse`` ``[B, Hq, Sq]`` (or ``[Hq, total_q]`` when Q is packed)."""
    q = _np(q)
    k = _np(k)
    v = _np(v)
    d = q.shape[-1]
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(d)
    Hq = q.shape[-2]
    Hkv = k.shape[-2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    packed_q = cu_seqlens_q is not None
    cu_q = None if cu_seqlens_q is None else np.asarray(_np(cu_seqlens_q, np.int64))
    cu_k = None if cu_seqlens_k is None else np.asarray(_np(cu_seqlens_k, np.int64))
    bt = None if block_table is None else np.asarray(_np(block_table, np.int64))
    n_seq = (len(cu_q) - 1) if packed_q else q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    if packed_q:
        lse = np.full((Hq, q.shape[0]), -np.inf)
    else:
        lse = np.full((q.shape[0], Hq, q.shape[1]), -np.inf)
    kw = dict(scale=scale, causal=causal, window_left=window_left,
              window_right=window_right, softcap=softcap, keep_window=keep_window)
    for b in range(n_seq):
        if packed_q:
            q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
            qb = q[q0:q1]
        else:
            qb = q[b]
        Sq = qb.shape[0]
        if bt is not None:
            Sk = int(cu_k[b + 1] - cu_k[b])
            kb = gather_paged(k, bt[b], Sk)
            vb = gather_paged(v, bt[b], Sk)
        elif cu_k is not None:
            k0, k1 = int(cu_k[b]), int(cu_k[b + 1])
            kb, vb = k[k0:k1], v[k0:k1]
            Sk = k1 - k0
        else:
            kb, vb = k[b], v[b]
            Sk = kb.shape[0]
        for h in range(Hq):
            g = h // G
            z = None if zero_hold_states is None else _np(zero_hold_states)[b, h, :Sk]
            slope = None if alibi_slopes is None else float(_np(alibi_slopes)[h])
            o, l = attention_rows(qb[:, h, :], kb[:, g, :], vb[:, g, :], np.arange(Sq), Sq, Sk,
                                  mask_rows=_mask_for(mask, b, h, Sq, Sk), z=z, alibi_slope=slope, **kw)
            if packed_q:
                out[q0:q1, h, :] = o
                lse[h, q0:q1] = l
            else:
                out[b, :, h, :] = o
                lse[b, h, :] = l
    return out, lse
