"""GPU parity of fa_bwd (dq, dk, dv) against the fp64 backward oracle.

The kernels round P and dS to the input type before their products (as the
forward rounds P), so the bar is relative, derived from that rounding
(2^-9 for bf16, 2^-12 for fp16, per product term, accumulated in fp32):
per gradient tensor, L1 error <= 1e-2 of the reference's L1 norm, max error
<= 2e-2 of the reference's max magnitude (+1e-3), cosine >= 0.9995."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import backward as B
from parity_util import DEV, to_dev

pytestmark = pytest.mark.gpu


def _grad_compare(got, ref, name):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite"
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    rel_l1 = err.sum() / max(np.abs(ref).sum(), 1e-30)
    cos = (got * ref).sum() / max(np.sqrt((got * got).sum() * (ref * ref).sum()), 1e-30)
    assert rel_l1 <= 1e-2, f"{name}: relative L1 {rel_l1:.3e}"
    assert err.max() <= 2e-2 * scale + 1e-3, f"{name}: max {err.max():.3e} vs scale {scale:.3e}"
    if scale > 0:
        assert cos >= 0.9995, f"{name}: cosine {cos:.6f}"
    return rel_l1


def _run(case, seed=0, **over):
    import masked_flash_attention_gb300 as fa
    p = dict(case["params"])
    p.update(over)
    dp = to_dev(p)
    q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
    out, lse, ws = fa.fa_fwd(q, k, v, **dp)
    g = torch.Generator().manual_seed(1000 + seed)
    dout = torch.randn(case["q"].shape, generator=g, dtype=torch.float32).to(case["q"].dtype)
    dq, dk, dv, ws2 = fa.fa_bwd(q, k, v, out, lse, dout.to(DEV), **dp)
    torch.cuda.synchronize()
    for w in (ws, ws2):
        rc, info = fa.fa_check_device_error(w)
        assert rc == 0, (rc, info)
    return dout, dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def check(case, seed=0, **over):
    dout, dq, dk, dv = _run(case, seed, **over)
    p = dict(case["params"])
    p.update(over)
    rq, rk, rv = B.attention_grad(case["q"], case["k"], case["v"], dout, **p)
    for got, ref, nm in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _grad_compare(got, ref, f"{case['name']}:{nm}")


CASES = [
    (2, 300, 300, 4, 2, 128, dict(causal=True)),                                   # self-attention, GQA
    (1, 200, 700, 8, 2, 128, dict(causal=True)),                                   # past KV
    (2, 256, 500, 4, 4, 64, dict(causal=False)),
    (1, 300, 600, 8, 4, 128, dict(causal=True, window_left=100, softcap=20.0)),
    (1, 400, 150, 4, 1, 64, dict(causal=True)),                                    # rows with no key
    (1, 1024, 1024, 8, 8, 128, dict(causal=True)),                                 # several tiles
    (1, 130, 260, 4, 2, 128, dict(causal=False, window_left=40, window_right=30)),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_backward(i):
    Bt, Sq, Sk, Hq, Hkv, d, extra = CASES[i]
    check(W.random_case(1400 + i, B=Bt, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra), seed=i)


def test_backward_varlen():
    q, k, v, cu_q, cu_k = W.random_varlen(1410, 4, 200, 400, 8, 2, 128, min_q=1)
    lq = int((cu_q[1:] - cu_q[:-1]).max())
    lk = int((cu_k[1:] - cu_k[:-1]).max())
    params = W.base_params(scale=128 ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=max(1, lq),
                           max_seqlen_k=max(1, lk), causal=True)
    check(dict(name="bwd_varlen", q=q, k=k, v=v, params=params))


def test_backward_alibi():
    c = W.random_case(1411, B=1, Sq=256, Sk=400, Hq=4, Hkv=2, d=128, causal=True)
    check(c, alibi_slopes=torch.tensor([0.5, 0.25, 0.125, 0.0625], dtype=torch.float32))


def test_backward_f16():
    c = W.random_case(1412, B=2, Sq=200, Sk=330, Hq=4, Hkv=2, d=128, causal=True, dtype=torch.float16)
    check(c)


def test_backward_decode_shape():
    # few query rows: the forward takes the split-KV path, the backward is the same
    c = W.random_case(1413, B=3, Sq=2, Sk=500, Hq=8, Hkv=2, d=128, causal=True, softcap=30.0)
    check(c)


def test_backward_deterministic():
    c = W.random_case(1414, B=1, Sq=300, Sk=300, Hq=4, Hkv=1, d=128, causal=True)
    a = _run(c)
    b = _run(c)
    for x, y in zip(a[1:], b[1:]):
        assert np.array_equal(x, y)


def test_backward_broadcast_kv_layout():
    # K/V broadcast over their heads (head stride 0)
    c = W.random_case(1415, B=2, Sq=150, Sk=300, Hq=4, Hkv=2, d=64, causal=True)
    k1, v1 = c["k"][:, :, :1], c["v"][:, :, :1]
    c = dict(c, k=k1.expand(-1, -1, 2, -1), v=v1.expand(-1, -1, 2, -1))
    check(c)


def test_backward_varlen_with_empty_sequences():
    # sequences without query rows, without keys, and ordinary ones
    g = torch.Generator().manual_seed(1416)
    lq = torch.tensor([0, 37, 130, 5, 0])
    lk = torch.tensor([40, 0, 260, 5, 0])
    cu_q = torch.zeros(6, dtype=torch.int32)
    cu_k = torch.zeros(6, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(lq, 0)
    cu_k[1:] = torch.cumsum(lk, 0)
    q = torch.randn(int(cu_q[-1]), 4, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(int(cu_k[-1]), 2, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(int(cu_k[-1]), 2, 128, generator=g).to(torch.bfloat16)
    params = W.base_params(scale=128 ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=130,
                           max_seqlen_k=260, causal=True)
    check(dict(name="bwd_varlen_empty", q=q, k=k, v=v, params=params))
