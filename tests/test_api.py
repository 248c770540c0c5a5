"""Host-side tests of the C ABI (no GPU work): the library loads, exports every
function include/fa.h declares, and the planner validates arguments with the
documented status codes (InfiniTrain pull request 193: an unsupported or
ill-formed call must report an error, never fall back)."""
import ctypes
import os
import re

import pytest
import torch

import masked_flash_attention_gb300 as fa
from masked_flash_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BF = torch.bfloat16


def header_functions():
    txt = open(os.path.join(ROOT, "include", "fa.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*|size_t)\s+(fa_\w+)\s*\(", txt, flags=re.M)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert "fa_fwd" in names and len(names) >= 6
    for n in names:
        assert hasattr(fa.lib, n), n
        assert ctypes.cast(getattr(fa.lib, n), ctypes.c_void_p).value
    assert fa.fa_abi_version() == 8 == _lib.ABI_VERSION
    assert fa.fa_status_string(0) == "ok"


def T(*shape, dtype=BF):
    return torch.zeros(*shape, dtype=dtype)


def plan(q, k, v, **kw):
    return fa.fa_fwd_plan(q, k, v, **kw)


def test_plan_ok_and_geometry():
    rc, p = plan(T(4, 1, 32, 128), T(4, 700, 8, 128), T(4, 700, 8, 128), causal=True)
    assert rc == 0
    assert p["path"] == _lib.FA_PATH_DECODE
    assert p["n_heads_sched"] == 8 and p["rows_per_tile"] == 8 and p["n_row_tiles"] == 1
    assert p["n_k_tiles"] == 6 and p["n_items"] == 32
    assert p["workspace_bytes"] >= p["off_tiles"] + 32 * 6 * 4


@pytest.mark.parametrize("hq,hkv,ok", [(12, 12, True), (32, 8, True), (16, 1, True),
                                       (12, 5, False), (8, 16, False)])
def test_head_rule(hq, hkv, ok):
    rc, _ = plan(T(1, 4, hq, 64), T(1, 8, hkv, 64), T(1, 8, hkv, 64))
    assert (rc == 0) == ok
    if not ok:
        assert rc == _lib.FA_ERR_INVALID_ARG


def test_invalid_arguments():
    q, k = T(1, 4, 2, 64), T(1, 8, 2, 64)
    E = _lib.FA_ERR_INVALID_ARG
    assert plan(q.float(), k, k)[0] == E                       # dtype
    assert plan(T(1, 4, 2, 96), T(1, 8, 2, 96), T(1, 8, 2, 96))[0] == E  # head dim
    assert plan(q, k, T(1, 9, 2, 64))[0] == E                  # K/V mismatch
    assert plan(q, k, k, window_left=-2)[0] == E
    assert plan(q, k, k, softcap=-1.0)[0] == E
    assert plan(q, k, k, softcap=float("inf"))[0] == E
    assert plan(q, k, k, scale=float("nan"))[0] == E
    assert plan(q, T(2, 8, 2, 64), T(2, 8, 2, 64))[0] == E     # batch mismatch
    qt = T(1, 2, 4, 64).transpose(1, 2)                         # transposed view is fine
    assert plan(qt, k, k)[0] == 0
    qs = T(1, 4, 2, 128)[..., :64]                              # head dim must be contiguous
    assert plan(qs, k, k)[0] == 0 or plan(qs, k, k)[0] == E
    assert plan(T(1, 4, 2, 64)[..., ::2], k, k)[0] == E         # non-unit head-dim stride
    assert plan(q, k, k, out=T(1, 4, 2, 64).float())[0] == E    # out dtype
    H = torch.float16
    assert plan(q.half(), k, k)[0] == E                          # q fp16, k/v bf16
    assert plan(q, k.half(), k)[0] == E                          # k fp16 only
    assert plan(q.half(), k.half(), k.half(), out=T(1, 4, 2, 64))[0] == E  # out bf16
    assert plan(q.half(), k.half(), k.half(), out=T(1, 4, 2, 64, dtype=H))[0] == 0
    assert plan(q, k, k, lse=T(1, 2, 5, dtype=torch.float32))[0] == E  # lse shape


def test_mask_rules():
    q, k = T(2, 4, 2, 64), T(2, 8, 2, 64)
    m = T(4, 8, dtype=torch.float32)
    assert plan(q, k, k, mask=m)[0] == 0
    assert plan(q, k, k, mask=T(1, 2, 4, 8, dtype=torch.float32))[0] == 0
    assert plan(q, k, k, mask=T(4, 9, dtype=torch.float32))[0] == _lib.FA_ERR_INVALID_ARG
    assert plan(q, k, k, mask=m.to(BF))[0] == _lib.FA_ERR_INVALID_ARG
    z = T(2, 2, 8, dtype=torch.float32)
    assert plan(q, k, k, zero_hold_states=z, keep_window=2, causal=True)[0] == 0
    assert plan(q, k, k, zero_hold_states=z, keep_window=0)[0] == _lib.FA_ERR_INVALID_ARG
    assert plan(q, k, k, zero_hold_states=z, keep_window=2,
                window_left=3)[0] == _lib.FA_ERR_UNSUPPORTED
    # dense mask with a packed variable-length batch is not implemented
    qv, kv = T(5, 2, 64), T(9, 2, 64)
    cu = torch.tensor([0, 5], dtype=torch.int32)
    cuk = torch.tensor([0, 9], dtype=torch.int32)
    assert plan(qv, kv, kv, cu_seqlens_q=cu, cu_seqlens_k=cuk, max_seqlen_q=5, max_seqlen_k=9,
                mask=T(5, 9, dtype=torch.float32))[0] == _lib.FA_ERR_UNSUPPORTED


def test_varlen_and_paged_rules():
    qv, kv = T(7, 4, 128), T(20, 2, 128)
    cu = torch.tensor([0, 3, 7], dtype=torch.int32)
    cuk = torch.tensor([0, 12, 20], dtype=torch.int32)
    ok = dict(cu_seqlens_q=cu, cu_seqlens_k=cuk, max_seqlen_q=4, max_seqlen_k=12)
    assert plan(qv, kv, kv, **ok)[0] == 0
    bad = dict(ok, max_seqlen_q=0)
    assert plan(qv, kv, kv, **bad)[0] == _lib.FA_ERR_INVALID_ARG
    assert plan(qv, kv, kv, cu_seqlens_q=cu, cu_seqlens_k=torch.tensor([0, 1], dtype=torch.int32),
                max_seqlen_q=4, max_seqlen_k=12)[0] == _lib.FA_ERR_INVALID_ARG
    kc = T(6, 16, 2, 128)
    bt = torch.zeros(2, 3, dtype=torch.int32)
    assert plan(qv, kc, kc, block_table=bt, **ok)[0] == 0
    assert plan(qv, kc, kc, block_table=bt, **dict(ok, max_seqlen_k=49))[0] == _lib.FA_ERR_INVALID_ARG
    # a page table without key counts is an error
    assert plan(qv, kc, kc, block_table=bt, cu_seqlens_q=cu, max_seqlen_q=4)[0] == _lib.FA_ERR_INVALID_ARG


def test_fwd_rejects_cpu_tensors():
    with pytest.raises(fa.FaError):
        fa.fa_fwd(T(1, 1, 1, 64), T(1, 2, 1, 64), T(1, 2, 1, 64))


def test_empty_problem_plans_no_items():
    rc, p = plan(T(2, 0, 4, 64), T(2, 5, 4, 64), T(2, 5, 4, 64))
    assert rc == 0 and p["n_items"] == 0


def test_kvcache_plan_rules():
    """fa_fwd_kvcache_plan: cache + active keys always take the split-KV kernel;
    shapes of k_new / v_new follow q with Hkv heads; max_seqlen_k is required;
    cache_seqlens has one int32 per sequence."""
    E = _lib.FA_ERR_INVALID_ARG
    q, kn = T(5, 4, 64), T(5, 2, 64)
    cu = torch.tensor([0, 2, 5], dtype=torch.int32)
    cl = torch.tensor([10, 0], dtype=torch.int32)
    kc = T(8, 16, 2, 64)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    kv = dict(cu_seqlens_q=cu, block_table=bt, max_seqlen_q=3, max_seqlen_k=13)
    rc, p = fa.fa_fwd_kvcache_plan(q, kc, kc, kn, kn, cl, **kv)
    assert rc == 0 and p["path"] == _lib.FA_PATH_DECODE and p["n_heads_sched"] == 2
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, kn, kn, cl, **dict(kv, max_seqlen_k=0))[0] == E
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, T(5, 1, 64), T(5, 1, 64), cl, **kv)[0] == E   # heads
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, T(4, 2, 64), T(4, 2, 64), cl, **kv)[0] == E   # rows
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, kn.half(), kn.half(), cl, **kv)[0] == E        # dtype
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, kn, kn, cl[:1], **kv)[0] == E                  # lengths
    assert fa.fa_fwd_kvcache_plan(q, kc, kc, kn, kn, cl.long(), **kv)[0] == E               # int32
    # padded cache [n_seq, cap, Hkv, d], fixed-length q [B, Sq, Hq, d]
    rc, p = fa.fa_fwd_kvcache_plan(T(2, 3, 4, 64), T(2, 40, 2, 64), T(2, 40, 2, 64), T(2, 3, 2, 64),
                                   T(2, 3, 2, 64), cl, max_seqlen_k=13, append=True)
    assert rc == 0 and p["path"] == _lib.FA_PATH_DECODE
    assert fa.fa_fwd_kvcache_plan(T(2, 3, 4, 64), T(3, 40, 2, 64), T(3, 40, 2, 64), T(2, 3, 2, 64),
                                  T(2, 3, 2, 64), cl, max_seqlen_k=13)[0] == E            # batch


def test_bwd_plan_rules():
    """fa_bwd_plan: the forward's arguments plus dout / dq like q and dk / dv
    like k, one element type; three kernels; Delta in the workspace."""
    E = _lib.FA_ERR_INVALID_ARG
    q, k = T(2, 5, 4, 64), T(2, 7, 2, 64)
    lse = T(2, 4, 5, dtype=torch.float32)
    rc, p = fa.fa_bwd_plan(q, k, k, q, lse, q, causal=True)
    assert rc == 0 and p["n_kernels"] == 3
    rc2, p2 = fa.fa_fwd_plan(q, k, k, out=q, lse=lse, causal=True)
    assert p["workspace_bytes"] >= p2["workspace_bytes"] + 2 * 4 * 5 * 4
    assert fa.fa_bwd_plan(q, k, k, q, lse, T(2, 5, 4, 32), causal=True)[0] == E       # dout shape
    assert fa.fa_bwd_plan(q, k, k, q, lse, q.half(), causal=True)[0] == E             # dout dtype
    assert fa.fa_bwd_plan(q, k, k, q, lse, q, dk=T(2, 7, 4, 64))[0] == E             # dk heads
    assert fa.fa_bwd_plan(q, k, k, q, lse, q, dq=T(2, 5, 4, 64)[..., ::2])[0] == E   # dq head-dim stride


def test_binding_abi_matches_header():
    txt = open(os.path.join(ROOT, "include", "fa.h")).read()
    assert int(re.search(r"#define FA_ABI_VERSION (\d+)", txt).group(1)) == _lib.ABI_VERSION


def test_binding_requires_every_declared_function():
    """The binding refuses a library that lacks an entry point the header
    declares (an older build), instead of failing only when it is called."""
    assert sorted(_lib.EXPORTS) == header_functions()


def test_noalloc_refuses_workspace_and_events():
    """fa_fwd_noalloc takes no workspace and no timing events: passing them
    is an error, not silently ignored (checked before any device work)."""
    q = T(1, 4, 2, 64)
    for kw in (dict(workspace=T(256, dtype=torch.uint8)), dict(event_begin=object()), dict(event_end=object())):
        with pytest.raises(fa.FaError) as e:
            fa.fa_fwd_noalloc(q, q, q, out=q, lse=T(1, 2, 4, dtype=torch.float32), **kw)
        assert e.value.status == _lib.FA_ERR_INVALID_ARG


def test_topk_prefill_layout_rule():
    """The many-row top-k path gathers key rows from a view where row
    b * Sk + j holds key j of sequence b with its heads side by side: a
    batch-contiguous bshd layout is taken, a [B, H, S, d] layout passed as a
    transposed view is refused (FA_ERR_UNSUPPORTED; the few-row path takes
    any layout)."""
    q = T(1, 300, 2, 64)
    z = torch.zeros(1, 2, 300)
    k = T(1, 300, 2, 64)
    assert plan(q, k, k, causal=True, zero_hold_states=z, keep_window=50)[0] == 0
    kt = T(1, 2, 300, 64).transpose(1, 2)
    assert plan(q, kt, kt, causal=True, zero_hold_states=z, keep_window=50)[0] == _lib.FA_ERR_UNSUPPORTED
    qd = T(1, 2, 2, 64)   # few rows: decode path, any layout
    assert plan(qd, kt, kt, causal=True, zero_hold_states=z[:, :, :300], keep_window=50)[0] == 0


def test_debug_dump_size():
    # S and P (128 x 128 fp32 each) and one reference per row, per key tile
    assert fa.fa_debug_dump_bytes_of(0) == 0
    assert fa.fa_debug_dump_bytes_of(3) == 3 * (2 * 128 * 128 + 128) * 4


@pytest.mark.gpu
def test_attention_end_event():
    """event_attn_end is recorded after the attention kernel itself and before
    the decode path's split combine: begin <= attention end <= end, and the
    results do not depend on the events."""
    import workloads as W
    dev = torch.device("cuda:0")
    case = W.paged_varlen_decode(seed=3, n_seq=8)
    p = {k_: (v_.to(dev) if isinstance(v_, torch.Tensor) else v_) for k_, v_ in case["params"].items()}
    q, k, v = case["q"].to(dev), case["k"].to(dev), case["v"].to(dev)
    rc, plan = fa.fa_fwd_plan(q, k, v, **p)
    assert rc == 0 and plan["n_splits"] > 1, plan
    out0, lse0, ws = fa.fa_fwd(q, k, v, **p)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record()  # torch creates the event handles on their first record
    out1, lse1, _ = fa.fa_fwd(q, k, v, workspace=ws, event_begin=ev[0], event_attn_end=ev[1], event_end=ev[2], **p)
    torch.cuda.synchronize()
    t_attn, t_all = ev[0].elapsed_time(ev[1]), ev[0].elapsed_time(ev[2])
    assert 0.0 < t_attn <= t_all
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
