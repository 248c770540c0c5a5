"""The bench's useful-work count (kept (query row, key, q-head) triples, the
numerator of every TFLOP/s it reports) against the fp64 oracle's logits: a
triple is useful exactly when the oracle's final logit is finite."""
import numpy as np
import pytest
import torch

import bench
import workloads as W
from oracle import attention as O


def _oracle_pairs(case):
    p = case["params"]
    q, k = case["q"], case["k"]
    packed = p["cu_seqlens_q"] is not None
    Hq = q.shape[-2]
    G = Hq // k.shape[-2]
    n_seq = len(p["cu_seqlens_q"]) - 1 if packed else q.shape[0]
    kw = dict(scale=1.0, causal=p["causal"], window_left=p["window_left"], window_right=p["window_right"],
              keep_window=p["keep_window"])
    total = 0
    for b in range(n_seq):
        if packed:
            q0, q1 = int(p["cu_seqlens_q"][b]), int(p["cu_seqlens_q"][b + 1])
            k0, k1 = int(p["cu_seqlens_k"][b]), int(p["cu_seqlens_k"][b + 1])
            qb, kb = q[q0:q1], k[k0:k1]
        else:
            qb, kb = q[b], k[b]
        Sq, Sk = qb.shape[0], kb.shape[0]
        for h in range(Hq):
            m = None
            if p["mask"] is not None:
                mm = p["mask"] if p["mask"].dim() == 2 else p["mask"][b % p["mask"].shape[0], h % p["mask"].shape[1]]
                m = mm[:Sq, :Sk].numpy()
            z = None if p["zero_hold_states"] is None else p["zero_hold_states"][b, h].numpy()
            x = O.logits_rows(qb[:, h].double().numpy(), kb[:, h // G].double().numpy(), np.arange(Sq), Sq, Sk,
                              mask_rows=m, z=z, **kw)
            total += int(np.isfinite(x).sum())
    return total


CASES = [
    dict(B=2, Sq=37, Sk=90, Hq=4, Hkv=2, causal=True),
    dict(B=1, Sq=90, Sk=40, Hq=2, Hkv=1, causal=True),                          # rows with no key
    dict(B=2, Sq=50, Sk=70, Hq=2, Hkv=2, causal=False, window_left=9, window_right=4),
    dict(B=1, Sq=64, Sk=64, Hq=3, Hkv=1, causal=True, window_left=20),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_pairs_rules(i):
    c = W.random_case(900 + i, d=64, **CASES[i])
    assert bench.useful_pairs(c) == _oracle_pairs(c)


@pytest.mark.parametrize("per_head", [False, True])
def test_pairs_dense_mask(per_head):
    c = W.random_case(910, B=2, Sq=40, Sk=60, Hq=2, Hkv=1, d=64, causal=True, window_left=30)
    if per_head:
        m = torch.stack([W.random_dense_mask(911 + h, 40, 60) for h in range(2)])[None]
    else:
        m = W.random_dense_mask(911, 40, 60)
    c["params"]["mask"] = m
    assert bench.useful_pairs(c) == _oracle_pairs(c)


def test_pairs_topk():
    c = W.random_case(920, B=1, Sq=48, Sk=48, Hq=2, Hkv=2, d=64, causal=True)
    c["params"]["zero_hold_states"] = W.random_zero_hold_states(920, 1, 2, 48, ties=True)
    c["params"]["keep_window"] = 7
    assert bench.useful_pairs(c) == _oracle_pairs(c)


def test_pairs_varlen():
    q, k, v, cu_q, cu_k = W.random_varlen(930, 4, 50, 80, 4, 2, 64, min_q=0)
    params = W.base_params(scale=0.125, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, causal=True, window_left=25)
    c = dict(name="varlen", q=q, k=k, v=v, params=params)
    assert bench.useful_pairs(c) == _oracle_pairs(c)


def test_pairs_worked_example_workload():
    # the sliding-window decode workload: one query, a 700-key additive mask
    c = W.sliding_window_decode(seed=0)
    assert bench.useful_pairs(c) == _oracle_pairs(c)


@pytest.mark.parametrize("window_left", [-1, 0, 37])
def test_kv_window_bytes(window_left):
    """Decode's algorithmic bytes: the K and V rows of every key that some
    query row of its sequence may see (the oracle's pair rules)."""
    g = torch.Generator().manual_seed(940)
    n_seq, Hkv, d = 6, 2, 64
    lk = torch.randint(1, 200, (n_seq,), generator=g)
    cu_k = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_k[1:] = torch.cumsum(lk, 0)
    cu_q = torch.arange(n_seq + 1, dtype=torch.int32)
    params = W.base_params(scale=0.125, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, causal=True,
                           window_left=window_left)
    case = dict(name="decode", q=torch.zeros(n_seq, 4, d, dtype=torch.bfloat16),
                k=torch.zeros(int(cu_k[-1]), Hkv, d, dtype=torch.bfloat16), v=None, params=params)
    want = 0
    for s in range(n_seq):
        Sk, Sq = int(lk[s]), 1
        ok = O.allowed_pairs(np.arange(Sq), np.arange(Sk), Sq, Sk, True, window_left, -1)
        want += int(ok.any(axis=0).sum()) * Hkv * d * 2 * 2
    assert bench.kv_window_bytes(case) == want


def test_l2_flush_rule():
    """Timed steps are separated by an L2 flush unless a step's own reads are
    several times L2 (the decode workloads); prefill and backward steps always
    flush."""
    tensor = dict(metric_units=1.0, unit="TFLOP/s", bound="tensor", flops=1.0, bytes=None)
    small = dict(metric_units=0.1, unit="GB/s", bound="hbm", flops=1.0, bytes=bench.L2_BYTES * 2)
    large = dict(small, bytes=749_203_456)  # K/V bytes of the paged-decode workload
    assert bench.flushes_l2(tensor) and bench.flushes_l2(small)
    assert not bench.flushes_l2(large)
    assert bench.flushes_l2(large, bwd=True)
    assert bench.NO_FLUSH_READ_BYTES >= 4 * bench.L2_BYTES


def test_kernel_hash_ignores_comments_only():
    """The traffic table's key follows the kernels' code: a comment or white
    space edit keeps it, any code edit changes it."""
    src = 'int f(int a) {  // the sum\n  /* two\n lines */ return a + 1;\n}\n'
    assert bench.code_text(src) == bench.code_text("int f(int a) {\n return a + 1; }  // other words")
    assert bench.code_text(src) != bench.code_text("int f(int a) { return a + 2; }")
    for kernel in bench.KERNEL_SOURCES:
        assert len(bench.kernel_hash(kernel)) == 16
