"""fa_fwd_noalloc: the forward pass for callers that cannot allocate device
memory (allocator-free runtimes, plugins whose host forbids device
allocations, latency paths that must not touch an allocator).  Its scratch is
a static device array inside the library, so the caller passes only inputs
and outputs.  These tests call it through the C ABI and check it against
fa_fwd (which uses a caller-provided workspace) within the parity tolerances,
on two calls in a row, since the static scratch keeps the previous call's
contents; one case also goes straight to the fp64 oracle.  The file is
named to be collected last."""
import gc

import numpy as np
import pytest
import torch

import masked_flash_attention_gb300 as fa
import workloads as W
from parity_util import DEV, LSE_ABS, MAX_ABS, MEAN_ABS, compare, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def _against_fa_fwd(case):
    p = to_dev(case["params"])
    q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
    ref_o, ref_l, ws = fa.fa_fwd(q, k, v, **p)
    torch.cuda.synchronize()
    assert fa.fa_check_device_error(ws)[0] == 0
    ref_o = ref_o.float().cpu().numpy()
    ref_l = ref_l.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(ref_l.shape, float("nan"), dtype=torch.float32, device=DEV)
        fa.fa_fwd_noalloc(q, k, v, out=out, lse=lse, **p)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        l_ = lse.cpu().numpy()
        assert np.isfinite(o).all()
        err = np.abs(o - ref_o)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
        assert np.array_equal(l_ == -np.inf, ref_l == -np.inf)
        fin = np.isfinite(ref_l)
        if fin.any():
            assert np.abs(l_[fin] - ref_l[fin]).max() <= LSE_ABS


def test_noalloc_paged_decode_split_kv():
    # split-KV decode: the scratch holds the work list and the split partials
    _against_fa_fwd(W.paged_varlen_decode(seed=2, n_seq=8, max_len=3000))


def test_noalloc_causal_gqa_and_dense_mask():
    _against_fa_fwd(W.random_case(21, B=2, Sq=5, Sk=700, Hq=8, Hkv=2, d=128, causal=True))
    c = W.sliding_window_decode(seed=4)
    _against_fa_fwd(c)


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    # 128 sequences x 8 K/V heads, 8192 keys: the split-KV partials alone need
    # about 64 MiB.  K/V are one sequence broadcast by a zero batch stride;
    # the call is rejected on the host before any kernel runs.
    q = torch.zeros(128, 1, 32, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 8192, 8, 128, dtype=torch.bfloat16, device=DEV).expand(128, -1, -1, -1)
    rc, plan = fa.fa_fwd_plan(q, k, k)
    assert rc == 0 and plan["workspace_bytes"] > (32 << 20)
    out = torch.empty_like(q)
    lse = torch.empty(128, 32, 1, dtype=torch.float32, device=DEV)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_noalloc(q, k, k, out=out, lse=lse)
    assert e.value.status == fa._lib.FA_ERR_WORKSPACE


def test_noalloc_against_the_oracle():
    """Directly against the fp64 oracle (not only through fa_fwd), on a
    prefill case with a ragged tail and on the worked example's decode."""
    for case in (W.random_case(22, B=2, Sq=200, Sk=450, Hq=8, Hkv=2, d=128, causal=True),
                 W.sliding_window_decode(seed=5)):
        p = to_dev(case["params"])
        q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
        ref_o, ref_l = run_oracle(case)
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            lse = torch.full(ref_l.shape, float("nan"), dtype=torch.float32, device=DEV)
            fa.fa_fwd_noalloc(q, k, v, out=out, lse=lse, **p)
            torch.cuda.synchronize()
            compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, case["name"] + "_noalloc")


def test_noalloc_allocates_nothing():
    """The entry point's reason to exist: after one warm-up call (which also
    loads the kernels), further calls leave both torch's allocator and the
    device's free memory unchanged."""
    case = W.paged_varlen_decode(seed=3, n_seq=8, max_len=2500)
    p = to_dev(case["params"])
    q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=DEV)
    fa.fa_fwd_noalloc(q, k, v, out=out, lse=lse, **p)
    torch.cuda.synchronize()
    # tensors left by earlier tests must not be freed in the middle of the
    # measurement (that would lower the counts): collect first, then hold
    gc.collect()
    gc.disable()
    try:
        alloc0 = torch.cuda.memory_allocated(DEV)
        free0 = torch.cuda.mem_get_info(DEV)[0]
        for _ in range(5):
            fa.fa_fwd_noalloc(q, k, v, out=out, lse=lse, **p)
            torch.cuda.synchronize()
        alloc1 = torch.cuda.memory_allocated(DEV)
        free1 = torch.cuda.mem_get_info(DEV)[0]
    finally:
        gc.enable()
    assert alloc1 == alloc0
    assert free1 == free0


def test_noalloc_refuses_device_validation():
    """FA_DEBUG_VALIDATE reports only through the device error word, which
    this entry point clears and cannot return: the flag is refused."""
    case = W.random_case(23, B=1, Sq=3, Sk=300, Hq=4, Hkv=2, d=64, causal=True)
    p = to_dev(case["params"])
    q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
    out = torch.empty_like(q)
    lse = torch.empty(1, 4, 3, dtype=torch.float32, device=DEV)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_noalloc(q, k, v, out=out, lse=lse, debug_flags=fa.FA_DEBUG_VALIDATE, **p)
    assert e.value.status == fa._lib.FA_ERR_UNSUPPORTED
