"""Pins of the backward oracle (``oracle/backward.py``) on the CPU, against
what the forward definition fixes without retyping the gradient formulas:

  * central finite differences of L = sum(O * dO), with O from the pinned
    forward oracle, for every element of dQ, dK, dV on tiny inputs, over the
    features the backward takes (causal with q_len != kv_len, windows, the
    soft-cap, ALiBi, grouped-query heads, packed sequences, a row with no
    allowed key);
  * shift invariance: adding one vector to every key of a (sequence, K/V
    head) leaves the softmax unchanged, so its dK rows sum to zero (without
    the soft-cap, which depends on the raw dot products).
"""
import numpy as np
import pytest
import torch

from oracle import attention as O
from oracle import backward as B


def _loss(q, k, v, dout, **kw):
    o, _ = O.attention(q, k, v, **kw)
    return float((o * dout).sum())


def _fd_grad(x, f, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = f()
        x[i] = old - eps
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


CASES = [
    # shape kwargs, forward kwargs
    (dict(B=1, Sq=4, Sk=4, Hq=2, Hkv=2), dict(causal=True)),
    (dict(B=2, Sq=3, Sk=6, Hq=4, Hkv=2), dict(causal=True)),                         # bottom-right, GQA
    (dict(B=1, Sq=5, Sk=7, Hq=2, Hkv=1), dict(causal=False, window_left=2, window_right=1)),
    (dict(B=1, Sq=4, Sk=5, Hq=2, Hkv=1), dict(causal=True, softcap=0.7)),             # soft-cap
    (dict(B=1, Sq=4, Sk=6, Hq=2, Hkv=2), dict(causal=True, alibi_slopes=np.array([0.5, 0.125]))),
    (dict(B=1, Sq=5, Sk=3, Hq=2, Hkv=1), dict(causal=True)),                          # rows with no key
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_finite_differences(i):
    shp, kw = CASES[i]
    rng = np.random.default_rng(40 + i)
    d = 3
    q = rng.standard_normal((shp["B"], shp["Sq"], shp["Hq"], d))
    k = rng.standard_normal((shp["B"], shp["Sk"], shp["Hkv"], d))
    v = rng.standard_normal((shp["B"], shp["Sk"], shp["Hkv"], d))
    do = rng.standard_normal(q.shape)
    kw = dict(kw, scale=0.9)
    dq, dk, dv = B.attention_grad(q, k, v, do, **kw)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = _fd_grad(x, lambda: _loss(q, k, v, do, **kw))
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-7)


def test_finite_differences_packed_sequences():
    rng = np.random.default_rng(7)
    cu_q = np.array([0, 2, 5])
    cu_k = np.array([0, 4, 7])
    q = rng.standard_normal((5, 2, 3))
    k = rng.standard_normal((7, 1, 3))
    v = rng.standard_normal((7, 1, 3))
    do = rng.standard_normal(q.shape)
    kw = dict(causal=True, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, scale=0.8, window_left=2)
    dq, dk, dv = B.attention_grad(q, k, v, do, **kw)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = _fd_grad(x, lambda: _loss(q, k, v, do, **kw))
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-7)


def test_key_shift_invariance():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(2, 9, 4, 8, generator=g, dtype=torch.float64)
    k = torch.randn(2, 12, 2, 8, generator=g, dtype=torch.float64)
    v = torch.randn(2, 12, 2, 8, generator=g, dtype=torch.float64)
    do = torch.randn(2, 9, 4, 8, generator=g, dtype=torch.float64)
    _, dk, _ = B.attention_grad(q, k, v, do, causal=True, window_left=5)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
