"""Shared helpers of the GPU parity tests: run a case through the C ABI,
compute the oracle, compare with the stated tolerances."""
import numpy as np
import torch

import masked_flash_attention_gb300 as fa
from oracle import attention as O

# Tolerances for bf16 outputs against the fp64 oracle (max-abs, mean-abs on
# O; absolute on fp32 LSE).  Beside them, internal gates taken per (sequence,
# q-head) block of rows: relative L1 error of O and cosine similarity, so that
# an all-zero or garbage O cannot pass on long rows where |O| is itself below
# the max-abs bound, and one wrong head cannot hide among many good ones.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3
REL_L1 = 1e-2
COS_MIN = 0.9999

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def to_dev(params):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in params.items()}


def run_gpu(case, **over):
    p = dict(case["params"])
    p.update(over)
    out, lse, ws = fa.fa_fwd(case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV), **to_dev(p))
    torch.cuda.synchronize()
    rc, info = fa.fa_check_device_error(ws)
    assert rc == 0, f"device error {rc} info {info}"
    return out.float().cpu().numpy(), lse.cpu().numpy(), ws


def run_oracle(case, **over):
    p = dict(case["params"])
    p.update(over)
    return O.attention(case["q"], case["k"], case["v"], **p)


def lse_as_out_rows(lse, out_ndim):
    """LSE rearranged to O's row order: [B,H,S] -> [B,S,H]; [H,T] -> [T,H]."""
    return np.moveaxis(lse, -1, 1) if out_ndim == 4 else lse.T


def compare(out, lse, ref_o, ref_l, name="", cu_seqlens=None):
    """Assert the parity bar; returns a dict of the measured errors (the
    block gates report their worst block).  ``cu_seqlens`` splits a packed
    [T, H, d] output into its sequences."""
    assert out.shape == ref_o.shape, (out.shape, ref_o.shape)
    assert lse.shape == ref_l.shape, (lse.shape, ref_l.shape)
    assert np.isfinite(out).all(), f"{name}: non-finite O"
    assert not np.isnan(lse).any(), f"{name}: NaN LSE"
    empty_ref = ref_l == -np.inf
    empty_gpu = lse == -np.inf
    assert (empty_ref == empty_gpu).all(), f"{name}: fully-masked row sets differ " \
        f"({int(empty_ref.sum())} vs {int(empty_gpu.sum())})"
    assert np.isfinite(lse[~empty_gpu]).all(), f"{name}: +inf LSE"
    rows_empty = lse_as_out_rows(empty_gpu, out.ndim)
    assert (out[rows_empty] == 0).all(), f"{name}: fully-masked rows are not exactly 0"
    err = np.abs(out - ref_o)
    res = dict(max_abs=float(err.max()) if err.size else 0.0,
               mean_abs=float(err.mean()) if err.size else 0.0)
    assert res["max_abs"] <= MAX_ABS, f"{name}: max |dO| {res['max_abs']}"
    assert res["mean_abs"] <= MEAN_ABS, f"{name}: mean |dO| {res['mean_abs']}"
    fin = ~empty_ref
    if fin.any():
        res["lse_abs"] = float(np.abs(lse[fin] - ref_l[fin]).max())
        assert res["lse_abs"] <= LSE_ABS, f"{name}: max |dLSE| {res['lse_abs']}"
    res["rel_l1"], res["cos"] = 0.0, 1.0
    for key, sl in head_blocks(out.shape, cu_seqlens):
        g, r = out[sl].reshape(-1).astype(np.float64), ref_o[sl].reshape(-1)
        denom = np.abs(r).sum()
        if denom == 0:  # every row of the block is fully masked (checked above)
            continue
        rel = float(np.abs(g - r).sum() / denom)
        cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r) + 1e-300))
        res["rel_l1"] = max(res["rel_l1"], rel)
        res["cos"] = min(res["cos"], cos)
        assert rel <= REL_L1, f"{name}: relative L1 {rel} in block {key}"
        assert cos >= COS_MIN, f"{name}: cosine {cos} in block {key}"
    return res


def head_blocks(shape, cu_seqlens=None):
    """(key, index) of every (sequence, q-head) block of rows of an output
    shaped [B, S, H, d], or [T, H, d] packed by ``cu_seqlens`` (without it,
    one block per head)."""
    if len(shape) == 4:
        for b in range(shape[0]):
            for h in range(shape[2]):
                yield (b, h), (b, slice(None), h)
        return
    cu = [0, shape[0]] if cu_seqlens is None else [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        if cu[s + 1] == cu[s]:
            continue
        for h in range(shape[1]):
            yield (s, h), (slice(cu[s], cu[s + 1]), h)
