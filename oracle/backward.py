"""Gradients of the masked attention forward (backward pass) -- test
infrastructure.

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of the
benchmark may use this module; the CUDA library never does.

The pages name the step (InfiniTrain pull request 193, "FlashAttention native
backend": the FlashAttention-2 forward and backward kernels; "Framework 与
autograd": an autograd function around them) without formulas; the backward
of the forward in ``attention.py`` is plain calculus.  With the loss L and
dL/dO = dO, per (sequence, q-head h, K/V head g = h // G):

  P      the softmax of the final logits (``attention.py`` rules 1-5)
  dV_g = sum over the group's q-heads of P_h^T dO_h
  dP   = dO_h V_g^T
  dX   = P * (dP - rowsum(P * dP))             (softmax Jacobian; rowsum(P * dP)
                                                equals rowsum(dO * O))
  the logit transform x = scale * s, or x = cap * tanh(scale * s / cap) with
  the soft-cap, has dx/ds = scale, or scale * (1 - tanh^2(scale * s / cap));
  ALiBi and additive terms are constants and get no gradient here
  dS   = dX * dx/ds                            (0 where the pair is dropped)
  dQ_h = dS K_g,   dK_g = sum over the group's q-heads of dS^T Q_h.

A row whose keys are all dropped has P = 0 and contributes nothing.
"""
from __future__ import annotations

import numpy as np

from .attention import _np, logits_rows, softmax_rows


def attention_grad(q, k, v, dout, *, scale=None, causal=False, window_left=-1, window_right=-1,
                   softcap=0.0, cu_seqlens_q=None, cu_seqlens_k=None, alibi_slopes=None, **_unused):
    """``(dq, dk, dv)`` in fp64, shaped like ``q``, ``k``, ``v``.  Layouts as
    in ``attention.attention``: ``[B, S, H, d]``, or packed ``[total, H, d]``
    with ``cu_seqlens_q`` / ``cu_seqlens_k``."""
    q, k, v, dout = _np(q), _np(k), _np(v), _np(dout)
    d = q.shape[-1]
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(d)
    Hq, Hkv = q.shape[-2], k.shape[-2]
    G = Hq // Hkv
    packed = cu_seqlens_q is not None
    cu_q = None if cu_seqlens_q is None else _np(cu_seqlens_q, np.int64)
    cu_k = None if cu_seqlens_k is None else _np(cu_seqlens_k, np.int64)
    n_seq = len(cu_q) - 1 if packed else q.shape[0]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(n_seq):
        if packed:
            qs = slice(int(cu_q[b]), int(cu_q[b + 1]))
            ks = slice(int(cu_k[b]), int(cu_k[b + 1]))
            qb, kb, vb, ob = q[qs], k[ks], v[ks], dout[qs]
        else:
            qb, kb, vb, ob = q[b], k[b], v[b], dout[b]
        Sq, Sk = qb.shape[0], kb.shape[0]
        gq = np.zeros_like(qb)
        gk = np.zeros_like(kb)
        gv = np.zeros_like(vb)
        for h in range(Hq):
            g = h // G
            qh, kg, vg, doh = qb[:, h], kb[:, g], vb[:, g], ob[:, h]
            slope = None if alibi_slopes is None else float(_np(alibi_slopes)[h])
            x = logits_rows(qh, kg, np.arange(Sq), Sq, Sk, scale=scale, causal=causal,
                            window_left=window_left, window_right=window_right, softcap=softcap,
                            alibi_slope=slope)
            p, _ = softmax_rows(x)
            dp = doh @ vg.T
            dx = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            if softcap and softcap > 0:
                t = np.tanh(float(scale) * (qh @ kg.T) / float(softcap))
                dxds = float(scale) * (1.0 - t * t)
            else:
                dxds = float(scale)
            ds = dx * dxds
            gq[:, h] = ds @ kg
            gk[:, g] += ds.T @ qh
            gv[:, g] += p.T @ doh
        if packed:
            dq[qs], dk[ks], dv[ks] = gq, gk, gv
        else:
            dq[b], dk[b], dv[b] = gq, gk, gv
    return dq, dk, dv
