"""Pins of the fp64 CPU oracle against facts that do not come from the oracle
itself: the ExecuTorch worked example, torch's fp64 scaled-dot-product
attention (a library routine) for the plain causal / full cases, closed forms,
invariants, a scalar brute force on tiny inputs, and hand-derived kept sets of
flash-sparse-attention's minimal top-k example.  CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as O
from oracle import brute

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f64(t):
    return t.detach().double().numpy()


def sdpa64(q, k, v, causal=False, scale=None):
    """torch fp64 SDPA on bshd inputs (MHA only), returns bshd numpy."""
    qt = torch.as_tensor(q).double().transpose(1, 2)
    kt = torch.as_tensor(k).double().transpose(1, 2)
    vt = torch.as_tensor(v).double().transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o.transpose(1, 2).numpy()


def sdpa_lse64(q, k, causal=False, scale=None):
    qt = torch.as_tensor(q).double().transpose(1, 2)
    kt = torch.as_tensor(k).double().transpose(1, 2)
    d = qt.shape[-1]
    s = (qt @ kt.transpose(-1, -2)) * (scale if scale else 1.0 / math.sqrt(d))
    if causal:
        L = s.shape[-1]
        s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    return torch.logsumexp(s, dim=-1).numpy()


def run(case, **over):
    p = dict(case["params"])
    p.update(over)
    return O.attention(case["q"], case["k"], case["v"], **p)


# ---------------------------------------------------------------------------
# ExecuTorch worked example (sliding window by additive mask, -inf chunk)
# ---------------------------------------------------------------------------

def test_worked_example_mask_equals_slice(golden):
    g = golden("executorch_sliding_window.json")
    case = W.sliding_window_decode(seed=0)
    mask = case["params"]["mask"]
    kept = np.nonzero(np.isfinite(mask.numpy()[0]))[0]
    assert kept[0] == g["kept_first"] and kept[-1] == g["kept_last"]
    assert len(kept) == g["previous_positions"] + 1
    assert mask.shape[1] == g["kv_len"]
    out, lse = run(case)
    lo, hi = g["kept_first"], g["kept_last"] + 1
    ref = sdpa64(case["q"], case["k"][:, lo:hi], case["v"][:, lo:hi], scale=0.125)
    ref_lse = sdpa_lse64(case["q"], case["k"][:, lo:hi], scale=0.125)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], ref_lse[0, 0], rtol=0, atol=1e-12)
    # the first key chunk of the kernel that the page describes is all -inf
    x = O.logits_rows(f64(case["q"][0, :, 0]), f64(case["k"][0, :, 0]), [0], 1, 700,
                      scale=0.125, mask_rows=mask.numpy())
    assert np.all(x[0, :g["key_chunk"]] == -np.inf)
    assert not np.any(np.isnan(x))


def test_worked_example_window_form_equals_mask_form(golden):
    g = golden("executorch_sliding_window.json")
    case = W.sliding_window_decode(seed=1)
    out_mask, lse_mask = run(case)
    n = g["query_position"] + 1  # cache filled up to and including the query
    out_win, lse_win = O.attention(case["q"], case["k"][:, :n], case["v"][:, :n], scale=0.125,
                                   causal=True, window_left=g["previous_positions"])
    np.testing.assert_allclose(out_win, out_mask, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_win, lse_mask, rtol=0, atol=1e-12)


def test_fully_masked_row_is_zero_not_nan():
    case = W.sliding_window_decode(seed=0, all_masked=True)
    out, lse = run(case)
    assert np.all(out == 0.0)
    assert np.all(lse == -np.inf)
    # causal with more queries than keys: the first rows see no key at all
    c = W.random_case(3, B=1, Sq=6, Sk=3, Hq=2, Hkv=2, d=8, causal=True)
    out, lse = run(c)
    assert np.all(out[0, :3] == 0.0) and np.all(lse[0, :, :3] == -np.inf)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse[0, :, 3:]))


def _merge_by_lse(parts):
    """Rows of attention over disjoint key chunks combined by their
    log-sum-exp: L = log sum_c e^{L_c}, O = sum_c e^{L_c - L} O_c; a row that
    no chunk lets see a key stays O = 0, L = -inf."""
    lses = np.stack([l for _, l in parts])            # [chunks, B, H, S]
    L = np.logaddexp.reduce(lses, axis=0)
    out = np.zeros_like(parts[0][0])
    for o, l in parts:
        w = np.where(np.isfinite(L), np.exp(l - np.where(np.isfinite(L), L, 0.0)), 0.0)
        out += o * np.moveaxis(w, 1, 2)[..., None]    # [B, H, S] -> [B, S, H, 1]
    return out, L


@pytest.mark.parametrize("split,all_neginf_chunk,empty_rows", [
    (0.37, False, False),  # every row sees keys of both chunks
    (0.5, True, True),     # the first chunk is all -inf for every row
    (0.81, False, True),   # the first rows see no key of the second chunk
])
def test_key_chunks_merge_by_lse(split, all_neginf_chunk, empty_rows):
    """ExecuTorch PR 10466 "Summary": attention may be computed chunk by
    chunk along the keys, the softmax accumulated and rescaled at the end,
    and an all -inf chunk must not poison the result.  Attention over all
    keys equals the log-sum-exp merge of attention over two key chunks (each
    chunk the other keys masked to -inf), rows that see no key in one chunk
    included; the tail split of the prefill kernel and the decode combine
    rely on exactly this."""
    Sq, Sk = 9, 23
    c = W.random_case(77, B=2, Sq=Sq, Sk=Sk, Hq=4, Hkv=2, d=8, causal=True)
    m = int(round(split * Sk))
    base = np.zeros((Sq, Sk))
    if all_neginf_chunk:  # every key of the first chunk masked for every row
        base[:, :m] = -np.inf
    full_o, full_l = run(c, mask=torch.tensor(base))
    chunk_a, chunk_b = base.copy(), base.copy()
    chunk_a[:, m:] = -np.inf
    chunk_b[:, :m] = -np.inf
    parts = [run(c, mask=torch.tensor(chunk_a)), run(c, mask=torch.tensor(chunk_b))]
    assert ((parts[0][1] == -np.inf).any() or (parts[1][1] == -np.inf).any()) == empty_rows
    out, lse = _merge_by_lse(parts)
    assert np.all(np.isfinite(out))
    np.testing.assert_array_equal(lse == -np.inf, full_l == -np.inf)
    np.testing.assert_allclose(out, full_o, rtol=0, atol=1e-13)
    fin = np.isfinite(full_l)
    np.testing.assert_allclose(lse[fin], full_l[fin], rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Causal: library routine, lower-triangular mask, bottom-right alignment
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,T,H,d", [(0, 17, 2, 16), (1, 64, 3, 32)])
def test_causal_square_equals_sdpa_and_triangular_mask(seed, T, H, d):
    c = W.random_case(seed, B=2, Sq=T, Sk=T, Hq=H, Hkv=H, d=d, causal=True)
    out, lse = run(c)
    ref = sdpa64(c["q"], c["k"], c["v"], causal=True)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, sdpa_lse64(c["q"], c["k"], causal=True), rtol=0, atol=1e-12)
    tri = np.where(np.tril(np.ones((T, T), dtype=bool)), 0.0, -np.inf)
    out_m, lse_m = run(c, causal=False, mask=tri)
    np.testing.assert_allclose(out_m, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_m, lse, rtol=0, atol=1e-13)


def test_full_attention_equals_sdpa():
    c = W.random_case(5, B=2, Sq=5, Sk=23, Hq=3, Hkv=3, d=16)
    out, lse = run(c)
    np.testing.assert_allclose(out, sdpa64(c["q"], c["k"], c["v"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, sdpa_lse64(c["q"], c["k"]), rtol=0, atol=1e-12)


def test_bottom_right_alignment():
    T, c_ = 40, 13
    c = W.random_case(2, B=1, Sq=T, Sk=T, Hq=2, Hkv=2, d=16, causal=True)
    full, full_lse = run(c)
    # q_len = kv_len - c: the new queries are the LAST rows of the square problem
    out, lse = O.attention(c["q"][:, T - c_:], c["k"], c["v"], causal=True)
    np.testing.assert_allclose(out, full[:, T - c_:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, full_lse[:, :, T - c_:], rtol=0, atol=1e-13)
    # a top-left reading would have given the FIRST rows instead
    assert not np.allclose(out, full[:, :c_])
    # one query over past KV, causal: attends to every key
    o1, l1 = O.attention(c["q"][:, :1], c["k"], c["v"], causal=True)
    o2, l2 = O.attention(c["q"][:, :1], c["k"], c["v"], causal=False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=0)
    np.testing.assert_allclose(o1, sdpa64(c["q"][:, :1], c["k"], c["v"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Grouped-query heads
# ---------------------------------------------------------------------------

def test_gqa_equals_explicit_repeat(golden):
    c = W.random_case(4, B=2, Sq=9, Sk=21, Hq=8, Hkv=2, d=16, causal=True)
    out, lse = run(c)
    kr = c["k"].repeat_interleave(4, dim=2)
    vr = c["v"].repeat_interleave(4, dim=2)
    out_r, lse_r = O.attention(c["q"], kr, vr, causal=True)
    np.testing.assert_allclose(out, out_r, rtol=0, atol=0)
    np.testing.assert_allclose(lse, lse_r, rtol=0, atol=0)
    # and a head-to-group slip (h % Hkv) would not match the library routine
    full = sdpa64(c["q"][:, -1:], kr[:, :], vr[:, :])
    o1, _ = O.attention(c["q"][:, -1:], c["k"], c["v"])
    np.testing.assert_allclose(o1, full, rtol=0, atol=1e-12)
    for case in golden("infinitrain_head_rule.json")["cases"]:
        q = torch.zeros(1, 1, case["hq"], 8)
        k = torch.zeros(1, 2, case["hkv"], 8)
        if case["kind"] == "error":
            with pytest.raises(ValueError):
                O.attention(q, k, k)
        else:
            O.attention(q, k, k)


# ---------------------------------------------------------------------------
# Varlen and paged
# ---------------------------------------------------------------------------

def test_varlen_equals_per_sequence():
    q, k, v, cu_q, cu_k = W.random_varlen(7, n_seq=4, max_q=9, max_k=20, Hq=4, Hkv=2, d=16,
                                          min_q=1, min_k=1)
    out, lse = O.attention(q, k, v, causal=True, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                           window_left=5)
    for s in range(4):
        q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        o, l = O.attention(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], causal=True,
                           window_left=5)
        np.testing.assert_allclose(out[q0:q1], o[0], rtol=0, atol=0)
        np.testing.assert_allclose(lse[:, q0:q1], l[0], rtol=0, atol=0)


def test_paged_equals_contiguous_and_permutation_invariant():
    q, k, v, cu_q, cu_k = W.random_varlen(8, n_seq=3, max_q=4, max_k=50, Hq=4, Hkv=1, d=8,
                                          min_q=1, min_k=1)
    ref, ref_lse = O.attention(q, k, v, causal=True, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                               softcap=5.0)
    for seed in (1, 2):
        kc, vc, bt = W.paginate(k, v, cu_k, page_size=16, seed=seed)
        out, lse = O.attention(q, kc, vc, causal=True, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                               block_table=bt, softcap=5.0)
        np.testing.assert_allclose(out, ref, rtol=0, atol=0)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=0)


# ---------------------------------------------------------------------------
# Softcap, softmax invariants, closed forms
# ---------------------------------------------------------------------------

def test_softcap_limits_and_brute():
    c = W.random_case(9, B=1, Sq=4, Sk=11, Hq=2, Hkv=2, d=8)
    o0, l0 = run(c)
    o1, l1 = run(c, softcap=1e7)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)
    o2, l2 = run(c, softcap=0.7)
    assert not np.allclose(o2, o0)
    qb = f64(c["q"][0, :, 0]).tolist()
    kb = f64(c["k"][0, :, 0]).tolist()
    vb = f64(c["v"][0, :, 0]).tolist()
    bo, bl = brute.attention(qb, kb, vb, scale=c["params"]["scale"], softcap=0.7)
    np.testing.assert_allclose(o2[0, :, 0], np.array(bo), rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2[0, 0], np.array(bl), rtol=0, atol=1e-13)


def test_softmax_rows_sum_to_one_and_lse():
    c = W.random_case(10, B=1, Sq=12, Sk=30, Hq=1, Hkv=1, d=16)
    m = W.random_dense_mask(10, 12, 30)
    x = O.logits_rows(f64(c["q"][0, :, 0]), f64(c["k"][0, :, 0]), np.arange(12), 12, 30,
                      scale=0.25, mask_rows=m.numpy(), causal=True)
    p, lse = O.softmax_rows(x)
    nonempty = np.isfinite(x).any(axis=1)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p[nonempty].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p[~nonempty] == 0)
    for r in range(12):
        fin = x[r][np.isfinite(x[r])]
        want = math.log(math.fsum(math.exp(t) for t in fin)) if len(fin) else -math.inf
        assert lse[r] == pytest.approx(want, abs=1e-12) if len(fin) else lse[r] == -np.inf


def test_closed_form_uniform_scores():
    # identical keys => all allowed logits equal => O is the mean of the
    # allowed V rows and LSE = s + ln(count)
    g = torch.Generator().manual_seed(11)
    Sq, Sk, d = 6, 15, 8
    q = torch.randn(1, Sq, 1, d, generator=g).to(torch.bfloat16)
    krow = torch.randn(d, generator=g).to(torch.bfloat16)
    k = krow.expand(1, Sk, 1, d).contiguous()
    v = torch.randn(1, Sk, 1, d, generator=g).to(torch.bfloat16)
    wl = 4
    out, lse = O.attention(q, k, v, causal=True, window_left=wl, scale=0.5)
    off = Sk - Sq
    V = f64(v[0, :, 0])
    for i in range(Sq):
        lo, hi = max(0, i + off - wl), i + off
        n = hi - lo + 1
        s = 0.5 * float(np.dot(f64(q[0, i, 0]), f64(krow)))
        np.testing.assert_allclose(out[0, i, 0], V[lo:hi + 1].mean(axis=0), rtol=0, atol=1e-13)
        assert lse[0, 0, i] == pytest.approx(s + math.log(n), abs=1e-12)


def test_closed_form_single_key():
    c = W.random_case(12, B=1, Sq=5, Sk=9, Hq=1, Hkv=1, d=8)
    out, lse = run(c, causal=True, window_left=0)  # only the diagonal key
    off = 4
    for i in range(5):
        j = i + off
        np.testing.assert_allclose(out[0, i, 0], f64(c["v"][0, j, 0]), rtol=0, atol=0)
        s = c["params"]["scale"] * float(np.dot(f64(c["q"][0, i, 0]), f64(c["k"][0, j, 0])))
        assert lse[0, 0, i] == pytest.approx(s, abs=1e-13)


# ---------------------------------------------------------------------------
# Brute force on tiny inputs
# ---------------------------------------------------------------------------

def _brute_case(c, h=0, b=0, **kw):
    G = c["q"].shape[2] // c["k"].shape[2]
    qb = f64(c["q"][b, :, h]).tolist()
    kb = f64(c["k"][b, :, h // G]).tolist()
    vb = f64(c["v"][b, :, h // G]).tolist()
    return brute.attention(qb, kb, vb, **kw)


@pytest.mark.parametrize("seed", range(12))
def test_random_tiny_vs_brute(seed):
    rng = np.random.default_rng(seed)
    Sq, Sk = int(rng.integers(1, 6)), int(rng.integers(1, 8))
    causal = bool(rng.integers(0, 2))
    wl = int(rng.integers(-1, 4))
    wr = int(rng.integers(-1, 3))
    cap = float(rng.choice([0.0, 0.9, 3.0]))
    use_mask = bool(rng.integers(0, 2))
    c = W.random_case(seed, B=1, Sq=Sq, Sk=Sk, Hq=2, Hkv=1, d=4, causal=causal,
                      window_left=wl, window_right=wr, softcap=cap)
    mask = W.random_dense_mask(seed, Sq, Sk).numpy() if use_mask else None
    out, lse = run(c, mask=mask)
    for h in range(2):
        bo, bl = _brute_case(c, h=h, scale=c["params"]["scale"], causal=causal, window_left=wl,
                             window_right=wr, softcap=cap,
                             mask=None if mask is None else mask.tolist())
        np.testing.assert_allclose(out[0, :, h], np.array(bo).reshape(Sq, 4), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], np.array(bl), rtol=0, atol=1e-13)


def _per_head_masks(seed, B, H, Sq, Sk):
    """[B, H, Sq, Sk] fp32 masks whose (b, h) slices all differ (each slice
    drawn from its own seed, with some -inf and some finite biases)."""
    return torch.stack([torch.stack([W.random_dense_mask(seed + 31 * b + h, Sq, Sk, p_neg_inf=0.25)
                                     for h in range(H)]) for b in range(B)])


@pytest.mark.parametrize("form", ["full", "broadcast_batch", "broadcast_head"])
def test_per_batch_and_head_mask_against_brute(form):
    """The [B|1, Hq|1, q_len, kv_len] mask form: each (sequence, q-head) takes
    its own slice.  Checked against the scalar brute force run per (b, h)
    with that slice as a plain 2-D mask, on a grouped-query case (Hq = 4,
    Hkv = 2, B = 2) where every slice differs, so that swapping b and h, or
    indexing the mask by the K/V head instead of the q-head, fails.  The
    broadcast forms use stride-0 views (torch expand), as a caller would pass
    them (ExecuTorch pull request 10466, "Summary": a [q_len, kv_len] mask
    added to q@k; one per head is the same rule applied head by head)."""
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 3, 6, 4
    G = Hq // Hkv
    c = W.random_case(61, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, causal=True)
    if form == "full":
        m = _per_head_masks(61, B, Hq, Sq, Sk)
    elif form == "broadcast_batch":
        m = _per_head_masks(62, 1, Hq, Sq, Sk).expand(B, -1, -1, -1)
        assert m.stride(0) == 0
    else:
        m = _per_head_masks(63, B, 1, Sq, Sk).expand(-1, Hq, -1, -1)
        assert m.stride(1) == 0
    # no two (b, h) slices coincide where the form gives them their own
    flat = m.reshape(B * Hq, Sq * Sk).numpy()
    distinct = {tuple(np.nan_to_num(r, neginf=-1e300)) for r in flat}
    assert len(distinct) == {"full": B * Hq, "broadcast_batch": Hq, "broadcast_head": B}[form]
    out, lse = run(c, mask=m)
    for b in range(B):
        for h in range(Hq):
            bo, bl = brute.attention(f64(c["q"][b, :, h]).tolist(), f64(c["k"][b, :, h // G]).tolist(),
                                     f64(c["v"][b, :, h // G]).tolist(), scale=c["params"]["scale"],
                                     causal=True, mask=m[b, h].double().numpy().tolist())
            np.testing.assert_allclose(out[b, :, h], np.array(bo), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[b, h], np.array(bl), rtol=0, atol=1e-13)


def test_per_head_mask_catches_wrong_head_index():
    """The check above can fail: a mask read with the K/V head index
    (h // G) instead of the q-head differs from the oracle on the same
    inputs.  Planted on the CPU by handing the oracle the mis-indexed
    mask."""
    B, Hq, Hkv, Sq, Sk, d = 1, 4, 2, 3, 6, 4
    G = Hq // Hkv
    c = W.random_case(64, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d)
    m = _per_head_masks(64, B, Hq, Sq, Sk)
    wrong = m[:, [h // G for h in range(Hq)]]
    out, _ = run(c, mask=m)
    out_wrong, _ = run(c, mask=wrong)
    assert np.abs(out - out_wrong).max() > 1e-3


def test_every_zero_neginf_mask_4x4():
    """Every 0/-inf pattern of a 4x4 tile: rows with no kept key are exactly
    zero with LSE -inf, nothing is NaN; a stride-sample also matches the
    brute force."""
    c = W.random_case(13, B=1, Sq=4, Sk=4, Hq=1, Hkv=1, d=2)
    qb = f64(c["q"][0, :, 0]).tolist()
    kb = f64(c["k"][0, :, 0]).tolist()
    vb = f64(c["v"][0, :, 0]).tolist()
    for bits in range(1 << 16):
        m = np.array([0.0 if (bits >> t) & 1 else -np.inf for t in range(16)]).reshape(4, 4)
        out, lse = O.attention(c["q"], c["k"], c["v"], scale=0.5, mask=m)
        empty = ~np.isfinite(m).any(axis=1)
        assert not np.isnan(out).any() and not np.isnan(lse).any()
        assert np.all(out[0, empty, 0] == 0.0) and np.all(lse[0, 0, empty] == -np.inf)
        assert np.all(np.isfinite(lse[0, 0, ~empty]))
        if bits % 97 == 0:
            bo, bl = brute.attention(qb, kb, vb, scale=0.5, mask=m.tolist())
            np.testing.assert_allclose(out[0, :, 0], np.array(bo), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[0, 0], np.array(bl), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# Dynamic top-k mask
# ---------------------------------------------------------------------------

# z for flash-sparse-attention's minimal example; keys 0 and 3 tie on 0.5.
# Hand derivation with keep_window = 2, causal (row i sees keys 0..i):
#   row 0: {0}              -> keep {0}
#   row 1: {0, 1}           -> both (no more than 2 candidates)
#   row 2: {0, 1, 2}        -> z: 2.0 (key 2), 0.5 (key 0), -1 (key 1) -> {0, 2}
#   row 3: {0, 1, 2, 3}     -> 2.0 (key 2), then the 0.5 tie goes to key 0 -> {0, 2}
# Not causal: every row keeps {0, 2}.
FSA_Z = [0.5, -1.0, 2.0, 0.5]
FSA_KEPT_CAUSAL = [[0], [0, 1], [0, 2], [0, 2]]
FSA_KEPT_FULL = [[0, 2]] * 4


def test_fsa_minimal_example_kept_sets(golden):
    g = golden("fsa_minimal_example.json")
    n, W_ = g["seq"], g["keep_window"]
    assert g["key"] == n == 4 and W_ == 2
    z = np.array(FSA_Z)
    for causal, want in ((True, FSA_KEPT_CAUSAL), (False, FSA_KEPT_FULL)):
        ok = O.allowed_pairs(np.arange(n), np.arange(n), n, n, causal=causal)
        got = [list(O.topk_kept_row(z, ok[i], W_)) for i in range(n)]
        assert got == want
        assert brute.kept_sets(FSA_Z, n, n, W_, causal=causal) == want


def test_fsa_minimal_example_outputs_closed_form():
    # Q = 0 => every QK logit is 0, so the logits are the kept z values; V = I
    # => O row i is the probability vector of row i.
    n = 4
    q = torch.zeros(1, n, 1, n)
    k = torch.randn(1, n, 1, n, generator=torch.Generator().manual_seed(0))
    v = torch.eye(n).reshape(1, n, 1, n)
    z = torch.tensor(FSA_Z).reshape(1, 1, n)
    out, lse = O.attention(q, k, v, causal=True, zero_hold_states=z, keep_window=2, scale=1.0)
    for i, kept in enumerate(FSA_KEPT_CAUSAL):
        denom = sum(math.exp(FSA_Z[j]) for j in kept)
        want = [math.exp(FSA_Z[j]) / denom if j in kept else 0.0 for j in range(n)]
        np.testing.assert_allclose(out[0, i, 0], want, rtol=0, atol=1e-15)
        assert lse[0, 0, i] == pytest.approx(math.log(denom), abs=1e-15)


@pytest.mark.parametrize("seed", range(10))
def test_topk_vs_brute(seed):
    rng = np.random.default_rng(100 + seed)
    Sq = int(rng.integers(1, 9))
    Sk = int(rng.integers(Sq, 11)) if seed % 2 == 0 else int(rng.integers(1, 11))
    causal = bool(seed % 3 != 0)
    keep = int(rng.integers(1, 6))
    c = W.random_case(seed, B=1, Sq=Sq, Sk=Sk, Hq=1, Hkv=1, d=4, causal=causal, softcap=2.0)
    z = W.random_zero_hold_states(seed, 1, 1, Sk, ties=True)
    out, lse = run(c, zero_hold_states=z, keep_window=keep)
    bo, bl = _brute_case(c, scale=c["params"]["scale"], causal=causal, softcap=2.0,
                         z=z[0, 0].tolist(), keep_window=keep)
    np.testing.assert_allclose(out[0, :, 0], np.array(bo).reshape(Sq, 4), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.array(bl), rtol=0, atol=1e-13)


def _expiry_rows(z, q_len, kv_len, keep):
    """Per key j: the first query row at which j is no longer kept, from the
    counting definition (beaters among keys 0..i+off)."""
    off = kv_len - q_len
    e = []
    for j in range(kv_len):
        beaters = sorted(kk for kk in range(kv_len)
                         if kk != j and (z[kk] > z[j] or (z[kk] == z[j] and kk < j)))
        e.append(beaters[keep - 1] - off if len(beaters) >= keep else q_len)
    return e


@pytest.mark.parametrize("seed", range(8))
def test_topk_interval_reading(seed):
    """The kept set of key j (causal) is the row interval [j - off, e_j), with
    e_j = (keep-th smallest index among keys beating j) - off: the compact form
    the GPU scheduler relies on."""
    rng = np.random.default_rng(200 + seed)
    Sk = int(rng.integers(2, 24))
    Sq = int(rng.integers(1, Sk + 1))
    keep = int(rng.integers(1, 7))
    z = W.random_zero_hold_states(seed, 1, 1, Sk, ties=bool(seed % 2))[0, 0].numpy()
    e = _expiry_rows(z.tolist(), Sq, Sk, keep)
    off = Sk - Sq
    ok = O.allowed_pairs(np.arange(Sq), np.arange(Sk), Sq, Sk, causal=True)
    for i in range(Sq):
        kept = set(O.topk_kept_row(z, ok[i], keep).tolist())
        interval = {j for j in range(Sk) if j <= i + off and i < e[j]}
        assert kept == interval


def test_fsa_minimal_example_expiry():
    # hand-derived: key 0 is beaten only by key 2, so it is never dropped
    # (e = q_len = 4); key 1's second beater is key 2 -> dropped from row 2;
    # key 2 has no beater (e = 4); key 3's beaters are keys 0 (tie, lower
    # index) and 2 -> e = 2, before its first causal row 3: never kept.
    assert _expiry_rows(FSA_Z, 4, 4, 2) == [4, 2, 4, 2]


# ---------------------------------------------------------------------------
# Named workloads are well formed
# ---------------------------------------------------------------------------

def test_paged_decode_workload_shapes():
    c = W.paged_varlen_decode(seed=0, n_seq=5, max_len=300)
    p = c["params"]
    lens = c["kv_lens"]
    assert p["cu_seqlens_k"][-1] == lens.sum()
    bt = p["block_table"]
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(c["k"].shape[0]))
    for s in range(5):
        assert int((bt[s] >= 0).sum()) == (int(lens[s]) + 15) // 16
    out, lse = O.attention(c["q"], c["k"], c["v"], **p)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


# ---------------------------------------------------------------------------
# ALiBi (the ``alibi_slopes`` argument of the vLLM pull request 11277 call):
# with Q = 0 every score is 0, so the weights are e^(-s * distance) and the
# row sums are geometric series with a closed form.
# ---------------------------------------------------------------------------

def _geometric(s, n):
    """sum_{d=0}^{n-1} e^(-s d)"""
    return (1.0 - math.exp(-s * n)) / (1.0 - math.exp(-s))


def test_alibi_causal_closed_form():
    n, s = 9, 0.37
    q = torch.zeros(1, n, 1, 16)
    k = torch.randn(1, n, 1, 16, generator=torch.Generator().manual_seed(3))
    v = torch.zeros(1, n, 1, 16)
    v[0, :, 0, :n] = torch.eye(n)  # V row j = e_j: O row i = the weights themselves
    out, lse = O.attention(q, k, v, causal=True, alibi_slopes=np.array([s]))
    for i in range(n):
        z = _geometric(s, i + 1)
        assert abs(lse[0, 0, i] - math.log(z)) < 1e-12
        want = np.zeros(16)
        for j in range(i + 1):
            want[j] = math.exp(-s * (i - j)) / z
        np.testing.assert_allclose(out[0, i, 0], want, atol=1e-14)


def test_alibi_bottom_right_single_query():
    # one query over n keys, causal: it sits on the last key, distances 0..n-1
    n, s = 12, 0.21
    q = torch.zeros(1, 1, 2, 8)
    k = torch.randn(1, n, 1, 8, generator=torch.Generator().manual_seed(4))
    v = torch.randn(1, n, 1, 8, generator=torch.Generator().manual_seed(5))
    _, lse = O.attention(q, k, v, causal=True, alibi_slopes=np.array([s, 2 * s]))
    assert abs(lse[0, 0, 0] - math.log(_geometric(s, n))) < 1e-12
    assert abs(lse[0, 1, 0] - math.log(_geometric(2 * s, n))) < 1e-12


def test_alibi_non_causal_two_sided():
    n, s = 7, 0.5
    q = torch.zeros(1, n, 1, 8)
    k = torch.randn(1, n, 1, 8, generator=torch.Generator().manual_seed(6))
    v = torch.randn(1, n, 1, 8, generator=torch.Generator().manual_seed(7))
    _, lse = O.attention(q, k, v, alibi_slopes=np.array([s]))
    for i in range(n):
        # keys at or left of i: distances 0..i; right of i: 1..n-1-i
        z = _geometric(s, i + 1) + (_geometric(s, n - i) - 1.0)
        assert abs(lse[0, 0, i] - math.log(z)) < 1e-12


def test_alibi_zero_slope_is_no_bias():
    g = torch.Generator().manual_seed(8)
    q, k, v = (torch.randn(2, 5, 4, 16, generator=g).bfloat16() for _ in range(3))
    a, la = O.attention(q, k[:, :, :2], v[:, :, :2], causal=True)
    b, lb = O.attention(q, k[:, :, :2], v[:, :, :2], causal=True, alibi_slopes=np.zeros(4))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
