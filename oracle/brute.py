"""Pure-Python scalar brute force of masked attention -- test infrastructure.

Written independently of ``oracle.attention`` (no numpy, no sort): every
logit, every kept-key decision and every softmax sum is a scalar loop, so that
a slip in the vectorised oracle (a transposed operand, a wrong head index, an
off-by-one in a rule) shows up as a disagreement on tiny inputs.

The kept set of the dynamic top-k mask (flash-sparse-attention issue 11,
"[Integration Progress Report] Dynamic Mask Attention Integration into
FlashAttention", "Overview" and "Next Steps" 4) is decided here by counting,
for each candidate key, the candidates that beat it (larger value, or equal
value and lower index); the key is kept when fewer than ``keep_window`` beat
it.  The oracle uses a sort instead.
"""
from __future__ import annotations

import math


def _beats(zk, k, zj, j):
    return zk > zj or (zk == zj and k < j)


def attention(q, k, v, *, scale, causal=False, window_left=-1, window_right=-1,
              softcap=0.0, mask=None, z=None, keep_window=0):
    """One (sequence, head): ``q`` is a list of ``q_len`` rows, ``k`` and ``v``
    lists of ``kv_len`` rows (lists of floats).  ``mask`` is a list of rows of
    floats (may hold -inf); ``z`` a list of ``kv_len`` floats.  Returns
    ``(out rows, lse list)``."""
    q_len, kv_len = len(q), len(k)
    d = len(q[0]) if q_len else 0
    dv = len(v[0]) if kv_len else d
    off = kv_len - q_len
    out, lses = [], []
    for i in range(q_len):
        allowed = []
        for j in range(kv_len):
            ok = True
            if causal and not (j <= i + off):
                ok = False
            if window_left >= 0 and not (j >= i + off - window_left):
                ok = False
            if window_right >= 0 and not (j <= i + off + window_right):
                ok = False
            allowed.append(ok)
        if z is not None:
            kept = []
            for j in range(kv_len):
                if not allowed[j]:
                    kept.append(False)
                    continue
                n_beat = 0
                for kk in range(kv_len):
                    if kk != j and allowed[kk] and _beats(z[kk], kk, z[j], j):
                        n_beat += 1
                kept.append(n_beat < keep_window)
            allowed = kept
        x = []
        for j in range(kv_len):
            if not allowed[j]:
                x.append(-math.inf)
                continue
            s = 0.0
            for t in range(d):
                s += q[i][t] * k[j][t]
            s *= scale
            if softcap > 0:
                s = softcap * math.tanh(s / softcap)
            if mask is not None:
                s += mask[i][j]
            if z is not None:
                s += z[j]
            x.append(s)
        m = -math.inf
        for xv in x:
            if xv > m:
                m = xv
        if m == -math.inf:
            out.append([0.0] * dv)
            lses.append(-math.inf)
            continue
        w = [math.exp(xv - m) if xv != -math.inf else 0.0 for xv in x]
        total = 0.0
        for wv in w:
            total += wv
        row = [0.0] * dv
        for j in range(kv_len):
            if w[j] == 0.0:
                continue
            pj = w[j] / total
            for t in range(dv):
                row[t] += pj * v[j][t]
        out.append(row)
        lses.append(m + math.log(total))
    return out, lses


def kept_sets(z, q_len, kv_len, keep_window, causal=True):
    """Kept key sets per row of the top-k mask, by counting beaters."""
    off = kv_len - q_len
    res = []
    for i in range(q_len):
        cand = [j for j in range(kv_len) if (not causal) or j <= i + off]
        kept = []
        for j in cand:
            n_beat = sum(1 for kk in cand if kk != j and _beats(z[kk], kk, z[j], j))
            if n_beat < keep_window:
                kept.append(j)
        res.append(kept)
    return res
