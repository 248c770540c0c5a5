"""Pins of the two-source oracle (``oracle/kvcache.py``) on the CPU.

vLLM pull request 11277, the author's reply on aligning with the unified
``flash_attn_varlen_func`` interface (first point): cached and active K/V are
passed separately.  The pins tie that form to the already pinned single-source
definition and to hand-worked values:
  * splitting any sequence's keys into cached rows (scattered over pages, or
    in a padded cache) and active rows changes nothing;
  * a worked example fixes the order (cached keys first) and the causal rule
    over the active keys;
  * no cached keys = causal self-attention over the active keys;
  * the append places each active row right after the cached ones and touches
    nothing else.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as O
from oracle import kvcache as K


def _split_case(seed, n_seq, max_k, Hq, Hkv, d, page=None, cap_extra=0):
    """Full per-sequence keys, cut at a random point into cached + active rows."""
    g = torch.Generator().manual_seed(seed)
    kv_lens = torch.randint(1, max_k + 1, (n_seq,), generator=g)
    q_lens = torch.stack([torch.randint(1, int(L) + 1, (1,), generator=g)[0] for L in kv_lens])
    cache_lens = kv_lens - q_lens
    cu_k = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_k[1:] = torch.cumsum(kv_lens, 0)
    cu_q = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(q_lens, 0)
    kf = torch.randn(int(cu_k[-1]), Hkv, d, generator=g, dtype=torch.float64)
    vf = torch.randn(int(cu_k[-1]), Hkv, d, generator=g, dtype=torch.float64)
    q = torch.randn(int(cu_q[-1]), Hq, d, generator=g, dtype=torch.float64)
    # active rows: the last q_len rows of each sequence's keys
    act = torch.cat([torch.arange(int(cu_k[b]) + int(cache_lens[b]), int(cu_k[b + 1])) for b in range(n_seq)])
    k_new, v_new = kf[act], vf[act]
    # cached rows: the first cache_len rows, in pages or a padded cache
    cu_c = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_c[1:] = torch.cumsum(cache_lens, 0)
    cidx = torch.cat([torch.arange(int(cu_k[b]), int(cu_k[b]) + int(cache_lens[b])) for b in range(n_seq)]
                     + [torch.zeros(0, dtype=torch.int64)])
    kc_flat, vc_flat = kf[cidx], vf[cidx]
    if page is not None:
        k_cache, v_cache, bt = W.paginate(kc_flat, vc_flat, cu_c, page, seed=seed)
    else:
        cap = int(cache_lens.max()) + cap_extra
        k_cache = torch.zeros(n_seq, max(cap, 1), Hkv, d, dtype=torch.float64)
        v_cache = torch.zeros_like(k_cache)
        for b in range(n_seq):
            n = int(cache_lens[b])
            k_cache[b, :n] = kc_flat[int(cu_c[b]):int(cu_c[b]) + n]
            v_cache[b, :n] = vc_flat[int(cu_c[b]):int(cu_c[b]) + n]
        bt = None
    return dict(q=q, kf=kf, vf=vf, cu_k=cu_k, cu_q=cu_q, k_new=k_new, v_new=v_new, k_cache=k_cache,
                v_cache=v_cache, bt=bt, cache_lens=cache_lens.to(torch.int32))


@pytest.mark.parametrize("seed,page,extra", [
    (0, 16, dict(causal=True)),
    (1, 1, dict(causal=True, window_left=7, softcap=5.0)),
    (2, None, dict(causal=True)),
    (3, 3, dict(causal=False, window_left=4, window_right=2)),
    (4, None, dict(causal=True, alibi_slopes=np.array([0.5, 0.25, 0.125, 0.0625]))),
])
def test_split_into_cache_and_active_changes_nothing(seed, page, extra):
    c = _split_case(seed, n_seq=4, max_k=40, Hq=4, Hkv=2, d=8, page=page)
    got_o, got_l = K.attention_kvcache(c["q"], c["k_cache"], c["v_cache"], c["k_new"], c["v_new"],
                                       c["cache_lens"], cu_seqlens_q=c["cu_q"], block_table=c["bt"],
                                       scale=0.4, **extra)
    ref_o, ref_l = O.attention(c["q"], c["kf"], c["vf"], cu_seqlens_q=c["cu_q"], cu_seqlens_k=c["cu_k"],
                               scale=0.4, **extra)
    np.testing.assert_allclose(got_o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(got_l), np.isinf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(got_l[fin], ref_l[fin], rtol=0, atol=1e-12)


def test_worked_example_order_and_causal_rule():
    # one cached key, two active keys, all keys 0 (uniform scores); values 1,
    # 10, 100.  Row 0 sees the cached key and active key 0: O = 11/2,
    # LSE = ln 2.  Row 1 sees all three: O = 111/3, LSE = ln 3.
    q = np.ones((2, 1, 1))
    k_cache = np.zeros((1, 4, 1, 1))
    v_cache = np.zeros((1, 4, 1, 1))
    v_cache[0, 0, 0, 0] = 1.0
    k_new = np.zeros((2, 1, 1))
    v_new = np.array([10.0, 100.0]).reshape(2, 1, 1)
    cu_q = np.array([0, 2])
    o, l = K.attention_kvcache(q, k_cache, v_cache, k_new, v_new, np.array([1]), cu_seqlens_q=cu_q,
                               causal=True, scale=1.0)
    np.testing.assert_allclose(o[:, 0, 0], [5.5, 37.0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l[0], [math.log(2.0), math.log(3.0)], rtol=0, atol=1e-12)


def test_empty_cache_is_causal_self_attention():
    g = torch.Generator().manual_seed(7)
    q = torch.randn(2, 9, 4, 8, generator=g, dtype=torch.float64)
    kn = torch.randn(2, 9, 2, 8, generator=g, dtype=torch.float64)
    vn = torch.randn(2, 9, 2, 8, generator=g, dtype=torch.float64)
    k_cache = torch.zeros(2, 16, 2, 8, dtype=torch.float64)
    o, l = K.attention_kvcache(q, k_cache, k_cache, kn, vn, np.array([0, 0]), causal=True)
    ro, rl = O.attention(q, kn, vn, causal=True)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("page", [16, 5, None])
def test_append_places_active_rows_after_cached_ones(page):
    c = _split_case(11, n_seq=3, max_k=30, Hq=2, Hkv=2, d=4, page=page, cap_extra=30)
    kc0, vc0 = np.asarray(c["k_cache"]), np.asarray(c["v_cache"])
    if page is not None:
        # room for the appended rows: extra pages at the end of each table row
        n_pages = kc0.shape[0]
        bt = c["bt"].numpy()
        need = [(int(c["cache_lens"][b]) + int(c["cu_q"][b + 1] - c["cu_q"][b]) + page - 1) // page
                for b in range(3)]
        width = max(need)
        new_bt = np.full((3, width), -1, dtype=np.int64)
        nxt = n_pages
        for b in range(3):
            have = (int(c["cache_lens"][b]) + page - 1) // page
            new_bt[b, :have] = bt[b, :have]
            for j in range(have, need[b]):
                new_bt[b, j] = nxt
                nxt += 1
        pad = np.zeros((nxt - n_pages,) + kc0.shape[1:])
        kc0 = np.concatenate([kc0, pad + 7.0])
        vc0 = np.concatenate([vc0, pad - 7.0])
        bt = new_bt
    else:
        bt = None
    kc1, vc1 = K.append_kvcache(kc0, vc0, c["k_new"], c["v_new"], c["cache_lens"], cu_seqlens_q=c["cu_q"],
                                block_table=bt)
    touched = np.zeros(kc0.shape[:2], dtype=bool)
    for b in range(3):
        n = int(c["cu_k"][b + 1] - c["cu_k"][b])
        full_k = c["kf"][int(c["cu_k"][b]):int(c["cu_k"][b + 1])].numpy()
        full_v = c["vf"][int(c["cu_k"][b]):int(c["cu_k"][b + 1])].numpy()
        np.testing.assert_array_equal(K.cached_rows(kc1, b, n, bt), full_k)
        np.testing.assert_array_equal(K.cached_rows(vc1, b, n, bt), full_v)
        for j in range(int(c["cache_lens"][b]), n):
            if bt is not None:
                touched[bt[b][j // page], j % page] = True
            else:
                touched[b, j] = True
    np.testing.assert_array_equal(kc1[~touched], kc0[~touched])
    np.testing.assert_array_equal(vc1[~touched], vc0[~touched])
