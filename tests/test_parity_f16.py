"""GPU parity with fp16 inputs (InfiniTrain pull request 193, "FlashAttention
native backend": the FlashAttention-2 kernels it builds take FP16 and BF16):
the same kernels, instantiated for fp16 operands, P and output, against the
fp64 oracle on freshly drawn fp16 inputs (fp32 N(0, 1) rounded to fp16, so the
mantissa bits that bf16 lacks are exercised)."""
import numpy as np
import pytest
import torch

import workloads as W
from parity_util import DEV, compare, run_gpu, run_oracle
from test_parity import _sampled

pytestmark = pytest.mark.gpu

F16 = torch.float16


def check(case, **over):
    assert case["q"].dtype == F16
    out, lse, _ = run_gpu(case, **over)
    ref_o, ref_l = run_oracle(case, **over)
    return compare(out, lse, ref_o, ref_l, case["name"] + "_f16", cu_seqlens=case["params"].get("cu_seqlens_q"))


def _assert_path(case, path, **over):
    import masked_flash_attention_gb300 as fa
    p = dict(case["params"])
    p.update(over)
    rc, plan = fa.fa_fwd_plan(case["q"], case["k"], case["v"], **p)
    assert rc == 0 and plan["path"] == path, plan


def _f16(case):
    return dict(case, q=case["q"].to(F16), k=case["k"].to(F16), v=case["v"].to(F16))


def _slopes(H):
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)


# tcgen05 prefill path
PREFILL = [
    (1, 129, 129, 2, 1, 128, dict(causal=True)),
    (2, 300, 700, 6, 2, 64, dict(causal=True)),
    (1, 256, 1000, 8, 8, 64, dict(causal=False)),
    (2, 200, 600, 8, 2, 128, dict(causal=True, window_left=150, window_right=10)),
    (1, 500, 500, 4, 1, 128, dict(causal=True, softcap=20.0)),
    (3, 140, 4100, 16, 8, 128, dict(causal=True)),
]


@pytest.mark.parametrize("i", range(len(PREFILL)))
def test_prefill_f16(i):
    import masked_flash_attention_gb300 as fa
    B, Sq, Sk, Hq, Hkv, d, extra = PREFILL[i]
    c = W.random_case(1300 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, dtype=F16, **extra)
    _assert_path(c, fa._lib.FA_PATH_PREFILL)
    check(c)


def test_prefill_f16_dense_mask():
    import masked_flash_attention_gb300 as fa
    c = W.random_case(1310, B=2, Sq=260, Sk=500, Hq=4, Hkv=2, d=128, causal=False, dtype=F16)
    m = W.random_dense_mask(1310, 260, 500)
    m[:, :128] = float("-inf")
    m[5] = float("-inf")
    _assert_path(c, fa._lib.FA_PATH_PREFILL, mask=m)
    check(c, mask=m)


def test_prefill_f16_topk():
    c = W.random_case(1311, B=1, Sq=400, Sk=400, Hq=2, Hkv=2, d=128, causal=True, dtype=F16)
    z = W.random_zero_hold_states(1311, 1, 2, 400, ties=True)
    check(c, zero_hold_states=z, keep_window=100)


def test_prefill_f16_varlen():
    q, k, v, cu_q, cu_k = W.random_varlen(1312, 4, 300, 600, 8, 2, 128, min_q=60, dtype=F16)
    lq = int((cu_q[1:] - cu_q[:-1]).max())
    lk = int((cu_k[1:] - cu_k[:-1]).max())
    params = W.base_params(scale=128 ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=lq,
                           max_seqlen_k=max(1, lk), causal=True)
    check(dict(name="prefill_varlen", q=q, k=k, v=v, params=params))


def test_prefill_f16_alibi():
    c = W.random_case(1313, B=2, Sq=300, Sk=700, Hq=8, Hkv=2, d=128, causal=True, dtype=F16)
    check(c, alibi_slopes=_slopes(8))


# split-KV decode path (mma.sync)
DECODE = [
    (3, 1, 700, 8, 2, 128, dict(causal=True)),
    (2, 4, 300, 4, 4, 64, dict(causal=True, window_left=100, softcap=10.0)),
    (1, 2, 1500, 32, 8, 128, dict(causal=False)),
]


@pytest.mark.parametrize("i", range(len(DECODE)))
def test_decode_f16(i):
    import masked_flash_attention_gb300 as fa
    B, Sq, Sk, Hq, Hkv, d, extra = DECODE[i]
    c = W.random_case(1320 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, dtype=F16, **extra)
    _assert_path(c, fa._lib.FA_PATH_DECODE)
    check(c)


def test_decode_f16_dense_mask_alibi():
    c = W.random_case(1325, B=2, Sq=3, Sk=400, Hq=4, Hkv=2, d=128, causal=True, dtype=F16)
    m = W.random_dense_mask(1325, 3, 400)
    m[:, :128] = float("-inf")
    check(c, mask=m, alibi_slopes=_slopes(4))


@pytest.mark.parametrize("page", [16, 1])
def test_paged_decode_f16(page):
    # page 16: TMA copies; page 1: the cp.async fallback
    q, k, v, cu_q, cu_k = W.random_varlen(1330 + page, 4, 2, 900, 8, 2, 128, min_q=1, dtype=F16)
    params = W.base_params(scale=128 ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                           max_seqlen_q=int((cu_q[1:] - cu_q[:-1]).max()),
                           max_seqlen_k=max(1, int((cu_k[1:] - cu_k[:-1]).max())),
                           causal=True, softcap=30.0)
    case = dict(name=f"paged{page}", q=q, k=k, v=v, params=params)
    kc, vc, bt = W.paginate(k, v, cu_k, page, seed=page)
    paged = dict(case, k=kc, v=vc, params=dict(params, block_table=bt))
    out, lse, _ = run_gpu(paged)
    ref_o, ref_l = run_oracle(case)
    compare(out, lse, ref_o, ref_l, f"paged{page}_f16", cu_seqlens=case["params"]["cu_seqlens_q"])


def test_f16_results_differ_from_bf16_reading():
    # the same fp16 bits read as bf16 would give another answer: the fp16
    # kernels must not agree with a bf16 run on the reinterpreted tensors
    c = W.random_case(1340, B=1, Sq=256, Sk=256, Hq=2, Hkv=2, d=64, causal=True, dtype=F16)
    o16, _, _ = run_gpu(c)
    cb = dict(c, q=c["q"].view(torch.bfloat16), k=c["k"].view(torch.bfloat16),
              v=c["v"].view(torch.bfloat16))
    ob, _, _ = run_gpu(cb)
    assert np.abs(np.asarray(o16, np.float64) - np.nan_to_num(np.asarray(ob, np.float64))).max() > 0.1


# full-size workloads in fp16, sampled rows
def test_causal_prefill_past_kv_full_f16():
    _sampled(_f16(W.causal_prefill_past_kv(seed=0)))


def test_paged_varlen_decode_full_f16():
    check(_f16(W.paged_varlen_decode(seed=0)))
