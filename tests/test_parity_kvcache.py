"""GPU parity of fa_fwd_kvcache: keys from two sources (the cache, then the
step's active rows) with and without the append (vLLM pull request 11277, the
author's reply on aligning with the unified flash_attn_varlen_func interface,
first point), against the two-source oracle.  Every cache row that is not a
cached key holds NaN before the call, so a kernel that read an unused page
row, or the rows the append is about to write, would produce NaN."""
import numpy as np
import pytest
import torch

from oracle import kvcache as K
from parity_util import DEV, compare

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def _case(seed, n_seq, max_k, Hq, Hkv, d, page=16, q_max=1, dtype=BF16, min_cache=0, fixed_q=False,
          cache_lens=None):
    g = torch.Generator().manual_seed(seed)
    if fixed_q:
        q_lens = torch.full((n_seq,), q_max, dtype=torch.int64)
    else:
        q_lens = torch.randint(1, q_max + 1, (n_seq,), generator=g)
    if cache_lens is None:
        cache_lens = torch.randint(min_cache, max_k + 1, (n_seq,), generator=g)
    else:
        cache_lens = torch.as_tensor(cache_lens, dtype=torch.int64)
    kv_lens = cache_lens + q_lens
    cu_q = torch.zeros(n_seq + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(q_lens, 0)
    tq = int(cu_q[-1])

    def rnd(*shape):
        return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)

    q = rnd(tq, Hq, d)
    k_new, v_new = rnd(tq, Hkv, d), rnd(tq, Hkv, d)
    if page is not None:
        # pages for the cached rows and the rows the append will fill
        pages_per = [(int(kv_lens[b]) + page - 1) // page for b in range(n_seq)]
        n_pages = sum(pages_per) + 3
        perm = torch.randperm(n_pages, generator=g)
        k_cache = torch.full((n_pages, page, Hkv, d), float("nan"), dtype=dtype)
        v_cache = k_cache.clone()
        bt = torch.full((n_seq, max(pages_per)), -1, dtype=torch.int32)
        pos = 0
        for b in range(n_seq):
            for p in range(pages_per[b]):
                bt[b, p] = int(perm[pos])
                pos += 1
            n = int(cache_lens[b])
            kv_k, kv_v = rnd(n, Hkv, d), rnd(n, Hkv, d)
            for p in range((n + page - 1) // page):
                lo, hi = p * page, min(n, (p + 1) * page)
                k_cache[int(bt[b, p]), :hi - lo] = kv_k[lo:hi]
                v_cache[int(bt[b, p]), :hi - lo] = kv_v[lo:hi]
    else:
        cap = int(kv_lens.max()) + 5
        k_cache = torch.full((n_seq, cap, Hkv, d), float("nan"), dtype=dtype)
        v_cache = k_cache.clone()
        for b in range(n_seq):
            n = int(cache_lens[b])
            k_cache[b, :n] = rnd(n, Hkv, d)
            v_cache[b, :n] = rnd(n, Hkv, d)
        bt = None
    c = dict(q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
             cache_lens=cache_lens.to(torch.int32), cu_q=cu_q, bt=bt,
             max_q=int(q_lens.max()), max_k=int(kv_lens.max()))
    if fixed_q:  # [B, Sq, H, d] layouts instead of packed rows
        c["q"] = q.view(n_seq, q_max, Hq, d)
        c["k_new"] = k_new.view(n_seq, q_max, Hkv, d)
        c["v_new"] = v_new.view(n_seq, q_max, Hkv, d)
        c["cu_q"] = None
    return c


def _run(c, append=False, **kw):
    import masked_flash_attention_gb300 as fa
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    kc, vc = dev(c["k_cache"]), dev(c["v_cache"])
    out, lse, ws = fa.fa_fwd_kvcache(
        dev(c["q"]), kc, vc, dev(c["k_new"]), dev(c["v_new"]), dev(c["cache_lens"]),
        cu_seqlens_q=dev(c["cu_q"]), block_table=dev(c["bt"]), append=append,
        max_seqlen_q=c["max_q"], max_seqlen_k=c["max_k"],
        **{k: (dev(v) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()})
    torch.cuda.synchronize()
    rc, info = fa.fa_check_device_error(ws)
    assert rc == 0, (rc, info)
    return out.float().cpu().numpy(), lse.cpu().numpy(), kc.cpu(), vc.cpu()


def _oracle(c, **kw):
    return K.attention_kvcache(c["q"], c["k_cache"], c["v_cache"], c["k_new"], c["v_new"], c["cache_lens"],
                               cu_seqlens_q=c["cu_q"], block_table=c["bt"], **kw)


def _check(c, name, append=False, **kw):
    out, lse, kc, vc = _run(c, append=append, **kw)
    ro, rl = _oracle(c, **kw)
    compare(out, lse, ro, rl, name, cu_seqlens=c["cu_q"])
    return kc, vc


def _check_append(c, kc, vc):
    """The cache after the call: the active rows right after the cached ones,
    bit for bit, and every other row (NaN included) as it was."""
    rk, rv = K.append_kvcache(c["k_cache"], c["v_cache"], c["k_new"], c["v_new"], c["cache_lens"],
                              cu_seqlens_q=c["cu_q"], block_table=c["bt"])
    for got, ref in ((kc, rk), (vc, rv)):
        # the reference holds the input values exactly (bf16/fp16 -> fp64)
        ref_t = torch.from_numpy(ref).to(got.dtype)
        num = ~torch.isnan(ref_t)
        assert torch.equal(got[num], ref_t[num])
        assert torch.isnan(got[~num]).all()  # rows nobody writes keep their NaN


CASES = [
    # seed, n_seq, max_cache, Hq, Hkv, d, page, q_max, extra
    (0, 8, 700, 32, 8, 128, 16, 1, dict(causal=True)),                              # decode, TMA pages
    (1, 6, 500, 8, 2, 128, 16, 20, dict(causal=True, window_left=64, softcap=30.0)),  # multi-token
    (2, 5, 300, 4, 4, 64, 1, 7, dict(causal=True)),                                 # page 1: cp.async
    (3, 5, 300, 8, 1, 128, 8, 3, dict(causal=True)),                                # page 8: cp.async
    (4, 4, 400, 16, 4, 64, None, 5, dict(causal=True)),                             # padded cache
    (5, 4, 40, 8, 8, 128, 16, 70, dict(causal=True)),                               # several row tiles
]


@pytest.mark.parametrize("i", range(len(CASES)))
@pytest.mark.parametrize("append", [False, True])
def test_kvcache(i, append):
    seed, n, mk, Hq, Hkv, d, page, qm, extra = CASES[i]
    c = _case(100 + seed, n, mk, Hq, Hkv, d, page=page, q_max=qm)
    kc, vc = _check(c, f"kvcache{i}", append=append, **extra)
    if append:
        _check_append(c, kc, vc)
    else:
        assert kc.view(torch.int16).equal(c["k_cache"].view(torch.int16))
        assert vc.view(torch.int16).equal(c["v_cache"].view(torch.int16))


def test_kvcache_fixed_length_q_and_empty_cache():
    c = _case(120, 3, 64, 8, 2, 128, page=16, q_max=9, fixed_q=True, cache_lens=[0, 30, 55])
    _check_append(c, *_check(c, "kvcache_fixed", append=True, causal=True))


def test_kvcache_cache_len_on_chunk_and_tile_edges():
    c = _case(121, 6, 300, 8, 2, 128, page=16, q_max=3, cache_lens=[0, 16, 128, 127, 129, 256])
    _check_append(c, *_check(c, "kvcache_edges", append=True, causal=True))


def test_kvcache_f16_alibi():
    c = _case(122, 4, 600, 8, 2, 128, page=16, q_max=4, dtype=torch.float16)
    slopes = torch.tensor([2.0 ** (-(h + 1)) for h in range(8)], dtype=torch.float32)
    _check(c, "kvcache_f16_alibi", append=True, causal=True, alibi_slopes=slopes)


def test_kvcache_full_size_decode_with_append():
    # the paged-decode workload's shape: 64 sequences, up to 8192 cached keys,
    # page 16, Hq 32 / Hkv 8, d 128, window 4096, soft-cap 30, one new token each
    c = _case(123, 64, 8191, 32, 8, 128, page=16, q_max=1, min_cache=127)
    kc, vc = _check(c, "kvcache_full", append=True, causal=True, window_left=4096, window_right=0,
                    softcap=30.0)
    _check_append(c, kc, vc)


def test_kvcache_append_past_capacity_is_reported():
    import masked_flash_attention_gb300 as fa
    c = _case(124, 2, 100, 4, 2, 64, page=None, q_max=3, fixed_q=True, cache_lens=[20, 99])
    cap = c["k_cache"].shape[1]  # 99 + 3 + 5
    c["cache_lens"][1] = cap - 1  # its 3 active rows would run past the padded cache
    c["max_k"] = cap + 3
    kc, vc = c["k_cache"].to(DEV), c["v_cache"].to(DEV)
    _, _, ws = fa.fa_fwd_kvcache(c["q"].to(DEV), kc, vc, c["k_new"].to(DEV), c["v_new"].to(DEV),
                                 c["cache_lens"].to(DEV), append=True,
                                 max_seqlen_q=c["max_q"], max_seqlen_k=c["max_k"], causal=True)
    rc, info = fa.fa_check_device_error(ws)
    assert rc == fa._lib.FA_ERR_DEVICE_BOUNDS and info == 1
    # the rejected sequence's rows were not written
    assert torch.isnan(kc[1, cap - 1:].cpu()).all()


def test_paged_decode_ignores_stale_page_rows():
    """fa_fwd over a paged cache whose unused page rows hold NaN: the last
    chunk of each sequence reads only rows inside the sequence."""
    import workloads as W
    from parity_util import run_gpu, run_oracle
    c = W.paged_varlen_decode(seed=5, n_seq=8, max_len=900)
    kc, vc = c["k"].clone(), c["v"].clone()
    bt = c["params"]["block_table"]
    lens = c["kv_lens"]
    page = kc.shape[1]
    for b in range(len(lens)):
        L = int(lens[b])
        last = int(bt[b, (L - 1) // page])
        kc[last, (L - 1) % page + 1:] = float("nan")
        vc[last, (L - 1) % page + 1:] = float("nan")
    c2 = dict(c, k=kc, v=vc)
    out, lse, _ = run_gpu(c2)
    ro, rl = run_oracle(c)
    compare(out, lse, ro, rl, "stale_rows", cu_seqlens=c["params"].get("cu_seqlens_q"))


def test_kvcache_sequences_without_new_tokens():
    # packed q with zero-length sequences: nothing is read from or appended for them
    c = _case(125, 5, 300, 8, 2, 128, page=16, q_max=3)
    lens = torch.tensor([2, 0, 3, 0, 1], dtype=torch.int32)
    cu = torch.zeros(6, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    n = int(cu[-1])
    c["q"], c["k_new"], c["v_new"] = c["q"][:n], c["k_new"][:n], c["v_new"][:n]
    c["cu_q"] = cu
    c["max_q"] = 3
    c["max_k"] = int((c["cache_lens"].long() + lens.long()).max())
    _check_append(c, *_check(c, "kvcache_no_new_tokens", append=True, causal=True))
