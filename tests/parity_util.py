"""Shared helpers of the GPU parity tests: run a case through the C ABI,
compute the oracle, compare with the stated tolerances."""
import numpy as np
import torch

import masked_flash_attention_gb300 as fa
from oracle import attention as O

# Tolerances for bf16 outputs against the fp64 oracle (max-abs, mean-abs on
# O; absolute on fp32 LSE).  Beside them, internal gates: relative L1 error of
# O and per-(row-block) cosine similarity, so that an all-zero or garbage O
# cannot pass on long rows where |O| is itself below the max-abs bound.
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


def compare(out, lse, ref_o, ref_l, name=""):
    """Assert the parity bar; returns a dict of the measured errors."""
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
    denom = np.abs(ref_o).sum()
    if denom > 0:
        res["rel_l1"] = float(err.sum() / denom)
        assert res["rel_l1"] <= REL_L1, f"{name}: relative L1 {res['rel_l1']}"
        a = out.reshape(-1).astype(np.float64)
        b = ref_o.reshape(-1)
        cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
        res["cos"] = cos
        assert cos >= COS_MIN, f"{name}: cosine {cos}"
    return res


