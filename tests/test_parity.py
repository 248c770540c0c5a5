"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on
the same seeded inputs (small cases element by element; full-size workloads
on sampled rows)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as O
from parity_util import DEV, compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def check(case, **over):
    out, lse, _ = run_gpu(case, **over)
    ref_o, ref_l = run_oracle(case, **over)
    return compare(out, lse, ref_o, ref_l, case["name"], cu_seqlens=case["params"].get("cu_seqlens_q"))


# ---------------------------------------------------------------------------
# ExecuTorch worked example: 700-key cache, keys 515..575, -inf first chunk
# ---------------------------------------------------------------------------

def test_worked_example():
    check(W.sliding_window_decode(seed=0))


def test_worked_example_all_masked_row():
    case = W.sliding_window_decode(seed=0, all_masked=True)
    out, lse, _ = run_gpu(case)
    assert (out == 0).all() and (lse == -np.inf).all()


@pytest.mark.parametrize("all_masked", [False, True])
def test_worked_example_without_skipping(all_masked):
    """Every key tile computed, including the all -inf ones: the -inf guard of
    the running softmax alone must keep the result NaN-free and exact."""
    from masked_flash_attention_gb300 import FA_DEBUG_NO_SKIP
    case = W.sliding_window_decode(seed=3, all_masked=all_masked)
    res_out, res_lse, _ = run_gpu(case, debug_flags=FA_DEBUG_NO_SKIP)
    ref_o, ref_l = run_oracle(case)
    compare(res_out, res_lse, ref_o, ref_l, "no-skip")


# ---------------------------------------------------------------------------
# Shape / feature sweep (several tiles, ragged tails)
# ---------------------------------------------------------------------------

SWEEP = [
    # B, Sq, Sk, Hq, Hkv, d, extra params
    (1, 1, 1, 1, 1, 64, dict()),
    (2, 1, 17, 4, 1, 128, dict(causal=True)),
    (1, 1, 700, 8, 8, 64, dict(causal=True, window_left=60)),
    (3, 1, 1030, 32, 8, 128, dict(causal=True, softcap=30.0)),
    (2, 3, 300, 12, 4, 64, dict(causal=True)),
    (1, 5, 129, 6, 2, 128, dict(causal=True, window_left=7, window_right=2)),
    (2, 4, 260, 16, 2, 128, dict()),                       # group of 8, not causal
    (1, 17, 200, 3, 1, 64, dict(causal=True)),             # 17*3 packed rows: 7 row tiles
    (2, 130, 300, 4, 2, 128, dict(causal=True)),
    (1, 257, 257, 2, 2, 64, dict(causal=True)),
    (1, 200, 100, 2, 1, 128, dict(causal=True)),           # q_len > kv_len: empty rows
    (1, 64, 500, 4, 4, 128, dict(causal=False, window_left=100, window_right=100)),
    (1, 33, 33, 32, 1, 64, dict(causal=True, softcap=5.0)),  # MQA
    (2, 2, 4096, 32, 8, 128, dict(causal=True, window_left=1000)),
]


@pytest.mark.parametrize("i", range(len(SWEEP)))
def test_sweep(i):
    B, Sq, Sk, Hq, Hkv, d, extra = SWEEP[i]
    check(W.random_case(100 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra))


def test_custom_scale():
    check(W.random_case(7, B=1, Sq=9, Sk=300, Hq=4, Hkv=2, d=64, causal=True, scale=0.3))


def test_transposed_kv_layout():
    """Past K/V stored as [B, H, S, d] and passed as a transposed view (a
    zero-copy metadata change, FastChat pull request 2315)."""
    c = W.random_case(8, B=2, Sq=3, Sk=333, Hq=8, Hkv=2, d=128, causal=True)
    kt = c["k"].transpose(1, 2).contiguous().transpose(1, 2)
    vt = c["v"].transpose(1, 2).contiguous().transpose(1, 2)
    assert not kt.is_contiguous()
    c2 = dict(c, k=kt, v=vt)
    check(c2)


def test_deterministic():
    c = W.random_case(9, B=2, Sq=2, Sk=900, Hq=8, Hkv=2, d=128, causal=True)
    a = run_gpu(c)
    b = run_gpu(c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# Dense additive masks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,B,Sq,Sk,Hq,Hkv,d,causal", [
    (0, 1, 1, 700, 1, 1, 64, False),
    (1, 2, 5, 300, 4, 2, 128, False),
    (2, 1, 3, 520, 8, 8, 64, True),
])
def test_dense_mask(seed, B, Sq, Sk, Hq, Hkv, d, causal):
    c = W.random_case(seed, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, causal=causal)
    m = W.random_dense_mask(seed, Sq, Sk)
    m[:, :128] = float("-inf")          # an all -inf key tile
    m[0, :] = float("-inf")             # a fully masked row
    m[:, 256:384] = 0.0                 # an all-zero tile
    check(c, mask=m)


def test_dense_mask_per_head():
    c = W.random_case(4, B=2, Sq=2, Sk=260, Hq=4, Hkv=2, d=64)
    m = torch.stack([torch.stack([W.random_dense_mask(10 * b + h, 2, 260) for h in range(4)])
                     for b in range(2)])
    m[1, 2] = float("-inf")
    check(c, mask=m)


# ---------------------------------------------------------------------------
# Dynamic top-k mask
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,B,Sq,Sk,H,d,keep,causal,ties", [
    (0, 1, 4, 4, 1, 64, 2, True, False),        # flash-sparse-attention minimal example
    (1, 2, 3, 300, 4, 128, 50, True, True),
    (2, 1, 9, 1000, 2, 64, 300, True, False),
    (3, 1, 2, 700, 2, 128, 100, False, True),
    (4, 1, 1, 129, 1, 64, 200, True, False),    # keep_window larger than the row
    (5, 1, 40, 9000, 2, 128, 3000, True, True),  # more than 64 key buckets
])
def test_topk(seed, B, Sq, Sk, H, d, keep, causal, ties):
    c = W.random_case(seed, B=B, Sq=Sq, Sk=Sk, Hq=H, Hkv=H, d=d, causal=causal)
    z = W.random_zero_hold_states(seed, B, H, Sk, ties=ties)
    check(c, zero_hold_states=z, keep_window=keep)


# ---------------------------------------------------------------------------
# Varlen and paged
# ---------------------------------------------------------------------------

def _varlen_case(seed, n_seq, max_q, max_k, Hq, Hkv, d, **p):
    q, k, v, cu_q, cu_k = W.random_varlen(seed, n_seq, max_q, max_k, Hq, Hkv, d)
    lq = (cu_q[1:] - cu_q[:-1]).max().item()
    lk = (cu_k[1:] - cu_k[:-1]).max().item()
    params = W.base_params(scale=d ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                           max_seqlen_q=max(1, lq), max_seqlen_k=max(1, lk))
    params.update(p)
    return dict(name=f"varlen{seed}", q=q, k=k, v=v, params=params), cu_k


@pytest.mark.parametrize("seed,n_seq,max_q,max_k,Hq,Hkv,d,extra", [
    (0, 5, 3, 600, 8, 2, 128, dict(causal=True)),
    (1, 4, 1, 300, 4, 4, 64, dict(causal=True, window_left=50, softcap=10.0)),
    (2, 3, 20, 200, 2, 1, 128, dict(causal=False)),
    (3, 6, 2, 64, 4, 2, 64, dict(causal=True)),         # some sequences may be empty
])
def test_varlen(seed, n_seq, max_q, max_k, Hq, Hkv, d, extra):
    case, _ = _varlen_case(seed, n_seq, max_q, max_k, Hq, Hkv, d, **extra)
    check(case)


@pytest.mark.parametrize("page", [16, 1, 64])
def test_paged(page):
    case, cu_k = _varlen_case(11, 4, 2, 500, 8, 2, 128, causal=True, softcap=30.0)
    kc, vc, bt = W.paginate(case["k"], case["v"], cu_k, page, seed=page)
    paged = dict(case, k=kc, v=vc)
    paged["params"] = dict(case["params"], block_table=bt)
    out, lse, _ = run_gpu(paged)
    ref_o, ref_l = run_oracle(case)   # same sequences, contiguous
    compare(out, lse, ref_o, ref_l, "paged", cu_seqlens=case["params"]["cu_seqlens_q"])


def test_paged_decode_workload_small():
    c = W.paged_varlen_decode(seed=1, n_seq=8, max_len=2000)
    check(c)


def test_bad_page_index_is_reported():
    """An out-of-range page index is found on the device, recorded in the
    error word and skipped (no fault): the caller sees FA_ERR_DEVICE_BOUNDS."""
    import masked_flash_attention_gb300 as fa
    case, cu_k = _varlen_case(12, 2, 1, 100, 4, 2, 64, causal=True)
    kc, vc, bt = W.paginate(case["k"], case["v"], cu_k, 16, seed=1)
    bt[0, 0] = kc.shape[0] + 5
    p = dict(case["params"], block_table=bt)
    out, lse, ws = fa.fa_fwd(case["q"].to(DEV), kc.to(DEV), vc.to(DEV), **to_dev(p))
    rc, info = fa.fa_check_device_error(ws)
    assert rc == fa._lib.FA_ERR_DEVICE_BOUNDS and info == kc.shape[0] + 5
    assert fa.fa_check_device_error(ws)[0] == 0  # cleared


# ---------------------------------------------------------------------------
# Tail split: a persistent grid's last round that fills at most half the grid
# runs each of its units as two pieces over the halves of its key tiles,
# merged by LSE (ExecuTorch PR 10466 "Summary": chunks along the key
# dimension, softmax accumulated progressively and rescaled at the end)
# ---------------------------------------------------------------------------

def _tail_hq(unit_rows, grid):
    """Smallest even q-head count whose units overflow the grid by at most half of it."""
    hq = grid // unit_rows + 1
    hq += hq & 1
    assert grid < unit_rows * hq <= grid + grid // 2
    return hq


TAIL = [
    # B, Sq, Sk, d, group size, extra
    (1, 500, 1000, 128, 2, dict()),                                    # ragged last key tile, 4 + 4 tiles
    (2, 300, 1400, 128, 2, dict(causal=True, softcap=30.0)),           # causal over past keys, 5 + 5 tiles
    (1, 1024, 2048, 128, 4, dict(causal=True, window_left=600)),       # sliding window, 3 + 3 tiles
    (1, 640, 900, 128, 2, dict(causal=False, window_left=300, window_right=200)),  # 3 + 2 tiles
]


@pytest.mark.parametrize("i", range(len(TAIL)))
def test_prefill_tail_split(i):
    import masked_flash_attention_gb300 as fa
    B, Sq, Sk, d, G, extra = TAIL[i]
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    rt = (Sq + 127) // 128
    hq = _tail_hq(B * rt, grid)
    case = W.random_case(1900 + i, B=B, Sq=Sq, Sk=Sk, Hq=hq, Hkv=hq // G, d=d, **extra)
    p = to_dev(case["params"])
    q, k, v = case["q"].to(DEV), case["k"].to(DEV), case["v"].to(DEV)
    rc, plan = fa.fa_fwd_plan(q, k, v, **p)
    assert rc == 0 and plan["tail_units"] == B * rt * hq - grid, plan
    ref_o, ref_l = run_oracle(case)
    ws = None
    for rep in range(2):  # the second call reuses the workspace: the arrival counts are back at zero
        out, lse, ws = fa.fa_fwd(q, k, v, workspace=ws, **p)
        torch.cuda.synchronize()
        rc, info = fa.fa_check_device_error(ws)
        assert rc == 0, (rc, info)
        assert int(ws[16:256].count_nonzero()) == 0
        compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, f"{case['name']} call {rep}")


# ---------------------------------------------------------------------------
# Full-size workloads, sampled rows
# ---------------------------------------------------------------------------

def _sampled(case, n_rows=48, seed=0):
    """Run the GPU on the whole workload; compare sampled (b, h, i) rows with
    the oracle evaluated row by row.  Each sampled row is its own block for
    the relative-L1 and cosine gates."""
    out, lse, _ = run_gpu(case)
    p = dict(case["params"])
    q, k, v = case["q"], case["k"], case["v"]
    B, Sq, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    rng = np.random.default_rng(seed)
    rows = [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(Sq))) for _ in range(n_rows)]
    rows += [(0, 0, 0), (B - 1, Hq - 1, Sq - 1)]
    ro, rl, go, gl = [], [], [], []
    kw = {kk: p[kk] for kk in ("causal", "window_left", "window_right", "softcap", "keep_window")}
    for b, h, i in rows:
        Sk = k.shape[1]
        z = None if p["zero_hold_states"] is None else p["zero_hold_states"][b, h].numpy()
        o_, l_ = O.attention_rows(q[b, i:i + 1, h].double().numpy(), k[b, :, h // G].double().numpy(),
                                  v[b, :, h // G].double().numpy(), [i], Sq, Sk, scale=p["scale"],
                                  z=z, **kw)
        ro.append(o_[0]); rl.append(l_[0]); go.append(out[b, i, h]); gl.append(lse[b, h, i])
    n = len(rows)
    return compare(np.array(go)[:, None, None, :], np.array(gl)[:, None, None],
                   np.array(ro)[:, None, None, :], np.array(rl)[:, None, None], case["name"])


def test_causal_prefill_past_kv_full():
    _sampled(W.causal_prefill_past_kv(seed=0))


def test_gpt2_small_layer_full():
    _sampled(W.gpt2_small_layer(seed=0))


def test_llama3_8b_layer_full():
    _sampled(W.llama3_8b_layer(seed=0), n_rows=32)


def test_dynamic_topk_full():
    _sampled(W.dynamic_topk(seed=0), n_rows=24)


def test_paged_varlen_decode_full():
    check(W.paged_varlen_decode(seed=0))


# ---------------------------------------------------------------------------
# tcgen05 prefill path (many query rows per K/V head)
# ---------------------------------------------------------------------------

def _assert_prefill(case, **over):
    import masked_flash_attention_gb300 as fa
    p = dict(case["params"])
    p.update(over)
    rc, plan = fa.fa_fwd_plan(case["q"], case["k"], case["v"], **p)
    assert rc == 0 and plan["path"] == fa._lib.FA_PATH_PREFILL, plan


PREFILL = [
    (1, 129, 129, 2, 1, 128, dict(causal=True)),                  # ragged tail, GQA pair
    (2, 300, 700, 6, 2, 64, dict(causal=True)),                   # group of 3: one lone head
    (1, 384, 384, 4, 4, 128, dict(causal=True)),                  # MHA: pairs of row tiles, odd count
    (1, 256, 1000, 8, 8, 64, dict(causal=False)),
    (2, 200, 600, 8, 2, 128, dict(causal=True, window_left=150, window_right=10)),
    (1, 500, 500, 4, 1, 128, dict(causal=True, softcap=20.0)),
    (1, 1000, 1000, 2, 2, 64, dict(causal=True)),
    (1, 300, 120, 4, 2, 128, dict(causal=True)),                  # q_len > kv_len
    (3, 140, 4100, 16, 8, 128, dict(causal=True)),                # long past KV
]


@pytest.mark.parametrize("i", range(len(PREFILL)))
def test_prefill_sweep(i):
    B, Sq, Sk, Hq, Hkv, d, extra = PREFILL[i]
    c = W.random_case(300 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra)
    _assert_prefill(c)
    check(c)


@pytest.mark.parametrize("all_masked", [False, True])
def test_prefill_without_skipping(all_masked):
    from masked_flash_attention_gb300 import FA_DEBUG_NO_SKIP
    c = W.random_case(320, B=1, Sq=300, Sk=300, Hq=4, Hkv=2, d=128, causal=True)
    m = None
    if all_masked:
        m = torch.zeros(300, 300)
        m[:130] = float("-inf")
    _assert_prefill(c, mask=m)
    out, lse, _ = run_gpu(c, mask=m, debug_flags=FA_DEBUG_NO_SKIP)
    ref_o, ref_l = run_oracle(c, mask=m)
    compare(out, lse, ref_o, ref_l, "prefill no-skip")


def test_prefill_dense_mask():
    c = W.random_case(321, B=2, Sq=260, Sk=500, Hq=4, Hkv=2, d=128, causal=False)
    m = W.random_dense_mask(321, 260, 500)
    m[:, :128] = float("-inf")
    m[5] = float("-inf")
    m[:, 256:384] = 0.0
    _assert_prefill(c, mask=m)
    check(c, mask=m)


def test_prefill_dense_mask_per_head():
    c = W.random_case(322, B=1, Sq=200, Sk=300, Hq=4, Hkv=4, d=64, causal=True)
    m = torch.stack([W.random_dense_mask(40 + h, 200, 300, p_neg_inf=0.5) for h in range(4)])[None]
    m[0, 1, :, :200] = float("-inf")
    _assert_prefill(c, mask=m)
    check(c, mask=m)


@pytest.mark.parametrize("causal,ties,Sq,Sk", [(True, True, 400, 400), (True, False, 400, 400), (False, True, 400, 400),
                                              (True, True, 300, 457)])
def test_prefill_topk(causal, ties, Sq, Sk):
    c = W.random_case(323, B=1, Sq=Sq, Sk=Sk, Hq=2, Hkv=2, d=128, causal=causal)
    z = W.random_zero_hold_states(323, 1, 2, Sk, ties=ties)
    _assert_prefill(c, zero_hold_states=z, keep_window=100)
    check(c, zero_hold_states=z, keep_window=100)


@pytest.mark.parametrize("seed,q_eq_k", [(0, False), (1, True)])
def test_prefill_varlen(seed, q_eq_k):
    q, k, v, cu_q, cu_k = W.random_varlen(330 + seed, 4, 300, 600, 8, 2, 128, q_eq_k=q_eq_k, min_q=60)
    lq = int((cu_q[1:] - cu_q[:-1]).max())
    lk = int((cu_k[1:] - cu_k[:-1]).max())
    params = W.base_params(scale=128 ** -0.5, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=lq,
                           max_seqlen_k=max(1, lk), causal=True)
    case = dict(name=f"prefill_varlen{seed}", q=q, k=k, v=v, params=params)
    _assert_prefill(case)
    check(case)


# ---------------------------------------------------------------------------
# ALiBi slopes (vLLM pull request 11277's flash_attn_varlen_func argument):
# prefill and decode, with and without other additive terms
# ---------------------------------------------------------------------------

def _alibi_slopes(H):
    # the usual geometric head slopes 2^(-8 (h + 1) / H)
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)


ALIBI = [
    (2, 300, 700, 8, 2, 128, dict(causal=True)),                                    # prefill, past KV
    (1, 256, 600, 4, 4, 64, dict(causal=False, window_left=200, window_right=50)),  # two-sided distances
    (1, 200, 200, 4, 2, 128, dict(causal=True, softcap=20.0)),                      # after the soft-cap
    (2, 1, 900, 8, 2, 128, dict(causal=True, softcap=30.0)),                        # decode
    (3, 2, 300, 4, 4, 64, dict(causal=True)),                                       # decode, 2 rows
]


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(len(ALIBI)))
def test_alibi(i):
    B, Sq, Sk, Hq, Hkv, d, extra = ALIBI[i]
    c = W.random_case(900 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra)
    check(c, alibi_slopes=_alibi_slopes(Hq))


@pytest.mark.gpu
def test_alibi_with_dense_mask():
    # decode path: ALiBi and a dense mask together
    c = W.random_case(910, B=2, Sq=3, Sk=400, Hq=4, Hkv=2, d=128, causal=True)
    m = W.random_dense_mask(910, 3, 400)
    m[:, :128] = float("-inf")
    check(c, mask=m, alibi_slopes=_alibi_slopes(4))


@pytest.mark.gpu
@pytest.mark.parametrize("seed,Sq,Sk,d,per_head,extra", [
    (911, 260, 400, 128, False, dict(causal=True)),
    (912, 300, 300, 64, True, dict(causal=True, softcap=20.0)),
    (913, 200, 333, 128, True, dict(causal=False, window_left=150, window_right=40)),
])
def test_alibi_with_dense_mask_prefill(seed, Sq, Sk, d, per_head, extra):
    # prefill path: the ALiBi penalty and a dense mask on the same logits
    c = W.random_case(seed, B=1, Sq=Sq, Sk=Sk, Hq=4, Hkv=2, d=d, **extra)
    if per_head:
        m = torch.stack([W.random_dense_mask(seed + h, Sq, Sk, p_neg_inf=0.3) for h in range(4)])[None]
    else:
        m = W.random_dense_mask(seed, Sq, Sk)
    _assert_prefill(c, mask=m, alibi_slopes=_alibi_slopes(4))
    check(c, mask=m, alibi_slopes=_alibi_slopes(4))


@pytest.mark.gpu
def test_alibi_with_topk_on_prefill_is_unsupported():
    import masked_flash_attention_gb300 as fa
    c = W.random_case(914, B=1, Sq=260, Sk=400, Hq=4, Hkv=4, d=128, causal=True)
    z = W.random_zero_hold_states(914, 1, 4, 400, ties=False)
    with pytest.raises(fa.FaError) as e:
        run_gpu(c, zero_hold_states=z, keep_window=50, alibi_slopes=_alibi_slopes(4))
    assert e.value.status == fa._lib.FA_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_alibi_paged_decode():
    c = W.paged_varlen_decode(seed=3, n_seq=6, max_len=700)
    check(c, alibi_slopes=_alibi_slopes(c["q"].shape[-2]))


def test_alibi_slopes_checked():
    import masked_flash_attention_gb300 as fa
    q = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(fa.FaError):
        fa._lib._alibi(torch.zeros(3), q)  # wrong length (and not on a device)


# ---------------------------------------------------------------------------
# FA_DEBUG_VALIDATE: mask values checked on the device
# ---------------------------------------------------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_validate_dense_mask_values(bad):
    import masked_flash_attention_gb300 as fa
    c = W.random_case(920, B=1, Sq=200, Sk=300, Hq=2, Hkv=2, d=64, causal=False)
    m = W.random_dense_mask(920, 200, 300)
    m[150, 77] = bad
    p = to_dev(dict(c["params"], mask=m))
    q, k, v = c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV)
    _, _, ws = fa.fa_fwd(q, k, v, debug_flags=fa.FA_DEBUG_VALIDATE, **p)
    rc, info = fa.fa_check_device_error(ws)
    assert rc == fa._lib.FA_ERR_DEVICE_VALUE
    # -inf and finite values pass; without the flag nothing is checked
    m2 = W.random_dense_mask(920, 200, 300)
    _, _, ws = fa.fa_fwd(q, k, v, debug_flags=fa.FA_DEBUG_VALIDATE, **to_dev(dict(c["params"], mask=m2)))
    assert fa.fa_check_device_error(ws)[0] == 0
    _, _, ws = fa.fa_fwd(q, k, v, **p)
    assert fa.fa_check_device_error(ws)[0] == 0


@pytest.mark.gpu
def test_validate_topk_scores():
    import masked_flash_attention_gb300 as fa
    c = W.random_case(921, B=1, Sq=256, Sk=256, Hq=2, Hkv=2, d=64, causal=True)
    z = W.random_zero_hold_states(921, 1, 2, 256)
    z[0, 1, 40] = float("nan")
    p = to_dev(dict(c["params"], zero_hold_states=z, keep_window=32))
    _, _, ws = fa.fa_fwd(c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV), debug_flags=fa.FA_DEBUG_VALIDATE, **p)
    assert fa.fa_check_device_error(ws)[0] == fa._lib.FA_ERR_DEVICE_VALUE


# ---------------------------------------------------------------------------
# Mask-free prefill at shapes whose unit counts do not divide the SM count:
# ragged rows over past keys, square causal at d = 64, a sliding window, the
# soft-cap variant, and full rows of 8 key tiles each
# ---------------------------------------------------------------------------

UNEVEN = [
    (2, 1000, 1500, 16, 4, 128, dict(causal=True)),
    (4, 1024, 1024, 12, 12, 64, dict(causal=True)),
    (4, 700, 2000, 16, 4, 128, dict(causal=True, window_left=300)),
    (1, 1500, 1500, 32, 8, 128, dict(causal=True, softcap=20.0)),
    (1, 1024, 1024, 24, 24, 128, dict(causal=False)),
]


@pytest.mark.parametrize("i", range(len(UNEVEN)))
def test_prefill_uneven_units(i):
    import masked_flash_attention_gb300 as fa
    B, Sq, Sk, Hq, Hkv, d, extra = UNEVEN[i]
    c = W.random_case(1800 + i, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra)
    rc, plan = fa.fa_fwd_plan(c["q"], c["k"], c["v"], **c["params"])
    assert rc == 0 and plan["path"] == fa._lib.FA_PATH_PREFILL, plan
    check(c)


def test_prefill_alibi_repeat_on_one_workspace():
    """The ALiBi variant, called twice in a row on one workspace with the
    outputs poisoned in between: nothing left in the workspace by the first
    call may leak into the second."""
    import masked_flash_attention_gb300 as fa
    c = W.random_case(1810, B=1, Sq=1200, Sk=1600, Hq=32, Hkv=8, d=64, causal=True)
    slopes = _alibi_slopes(32)
    p = dict(c["params"], alibi_slopes=slopes)
    ref_o, ref_l = run_oracle(c, alibi_slopes=slopes)
    q, k, v = c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV)
    out, lse, ws = fa.fa_fwd(q, k, v, **to_dev(p))
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        fa.fa_fwd(q, k, v, out=out, lse=lse, workspace=ws, **to_dev(p))
        torch.cuda.synchronize()
        assert fa.fa_check_device_error(ws)[0] == 0
        compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "alibi repeat")
