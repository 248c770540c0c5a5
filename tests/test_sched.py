"""GPU tests of the tile scheduler: the work list it leaves in the workspace
against a classification recomputed on the CPU from the oracle's logits;
EMPTY tiles never appear (ExecuTorch pull request 10466 "Summary": a fully
-inf chunk need not be computed); top-k kept sets match the oracle exactly
(flash-sparse-attention issue 11 "Current Status": mask max/mean difference
0.0 and position match 1.0)."""
import numpy as np
import pytest
import torch

import masked_flash_attention_gb300 as fa
import workloads as W
from oracle import attention as O
from parity_util import DEV, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def worklist(case, **over):
    p = dict(case["params"])
    p.update(over)
    rc, plan = fa.fa_fwd_plan(case["q"], case["k"], case["v"], **p)
    assert rc == 0
    out, lse, ws = run_gpu(case, **over)
    w = ws.cpu()
    n, nk = plan["n_items"], plan["n_k_tiles"]
    counts = w[plan["off_counts"]:plan["off_counts"] + 4 * n].view(torch.int32).numpy()
    tiles = w[plan["off_tiles"]:plan["off_tiles"] + 4 * n * nk].view(torch.int32).numpy().reshape(n, nk)
    stats = w[plan["off_stats"]:plan["off_stats"] + 24].view(torch.int64).numpy()
    return plan, counts, tiles, stats, ws


def oracle_classes(case, plan, **over):
    """[n_items, n_k_tiles] classes from the oracle's logit matrices: EMPTY
    if every pair of the item's rows x the tile's keys is -inf; FULL if none
    is and no additive term is present; else PARTIAL."""
    p = dict(case["params"])
    p.update(over)
    q, k, v = case["q"], case["k"], case["v"]
    B, Sq, Hq, d = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    KT = plan["keys_per_tile"]
    n_rt, nk = plan["n_row_tiles"], plan["n_k_tiles"]
    decode = plan["path"] == fa._lib.FA_PATH_DECODE
    cls = np.zeros((plan["n_items"], nk), dtype=np.int32)
    z = p.get("zero_hold_states")
    m = p.get("mask")
    for b in range(B):
        for hs in range(plan["n_heads_sched"]):
            heads = range(hs * G, hs * G + G) if decode else [hs]
            X, M = [], []
            for h in heads:
                mh = None if m is None else (m.numpy() if m.dim() == 2 else m[b, h].numpy())
                x = O.logits_rows(q[b, :, h].double().numpy(), k[b, :, h // G].double().numpy(),
                                  np.arange(Sq), Sq, Sk, scale=p["scale"] or d ** -0.5,
                                  causal=p["causal"], window_left=p["window_left"],
                                  window_right=p["window_right"], softcap=p["softcap"],
                                  mask_rows=mh, z=None if z is None else z[b, h].numpy(),
                                  keep_window=p["keep_window"])
                X.append(x)
                M.append(np.zeros((Sq, Sk)) if mh is None else mh)
            X, M = np.stack(X), np.stack(M)
            for rt in range(n_rt):
                if decode:
                    R = plan["rows_per_tile"]  # packed rows (query, head-in-group)
                    i0, i1 = rt * R // G, (rt * R + R - 1) // G
                else:
                    i0, i1 = rt * plan["rows_per_tile"], (rt + 1) * plan["rows_per_tile"] - 1
                i1 = min(i1, Sq - 1)
                item = (b * plan["n_heads_sched"] + hs) * n_rt + rt
                for kt in range(nk):
                    blk = X[:, i0:i1 + 1, kt * KT:min(Sk, (kt + 1) * KT)]
                    mblk = M[:, i0:i1 + 1, kt * KT:min(Sk, (kt + 1) * KT)]
                    if blk.size == 0 or np.all(blk == -np.inf):
                        cls[item, kt] = 0
                    elif np.all(np.isfinite(blk)) and z is None and np.all(mblk == 0):
                        # nothing masked and no additive term: the tile needs no predicate
                        cls[item, kt] = 1
                    else:
                        cls[item, kt] = 2
    return cls


def gpu_classes(plan, counts, tiles):
    cls = np.zeros((plan["n_items"], plan["n_k_tiles"]), dtype=np.int32)
    for it in range(plan["n_items"]):
        seen = []
        for e in tiles[it, :counts[it]]:
            kt, part = int(e) >> 1, int(e) & 1
            seen.append(kt)
            cls[it, kt] = 2 if part else 1
        assert seen == sorted(set(seen)), "tiles must be listed once, in key order"
    return cls


def test_worked_example_schedules_one_partial_tile():
    case = W.sliding_window_decode(seed=0)
    plan, counts, tiles, stats, _ = worklist(case)
    assert plan["n_items"] == 1 and plan["n_k_tiles"] == 6
    assert counts[0] == 1 and tiles[0, 0] == (4 << 1) | 1   # keys 512..639 hold 515..575
    assert tuple(stats) == (0, 1, 5)
    # all -inf row: nothing scheduled at all
    plan, counts, tiles, stats, _ = worklist(W.sliding_window_decode(seed=0, all_masked=True))
    assert counts[0] == 0 and tuple(stats) == (0, 0, 6)


def test_no_skip_schedules_everything():
    case = W.sliding_window_decode(seed=0)
    plan, counts, tiles, stats, _ = worklist(case, debug_flags=fa.FA_DEBUG_NO_SKIP)
    assert counts[0] == 6 and tuple(stats) == (0, 6, 0)


@pytest.mark.parametrize("seed,B,Sq,Sk,Hq,Hkv,d,extra", [
    (0, 2, 3, 700, 8, 2, 64, dict(causal=True, window_left=200)),
    (1, 1, 9, 520, 4, 4, 64, dict(causal=True)),
    (2, 1, 5, 900, 6, 3, 128, dict(causal=False, window_left=130, window_right=0)),
])
def test_geometric_classes_exact(seed, B, Sq, Sk, Hq, Hkv, d, extra):
    case = W.random_case(seed, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra)
    plan, counts, tiles, stats, _ = worklist(case)
    got = gpu_classes(plan, counts, tiles)
    want = oracle_classes(case, plan)
    assert np.array_equal(got == 0, want == 0)           # EMPTY set exact
    assert np.all(want[got == 1] == 1)                    # FULL only where nothing is masked


def test_dense_mask_classes_exact():
    case = W.random_case(5, B=1, Sq=2, Sk=900, Hq=2, Hkv=2, d=64)
    m = torch.zeros(2, 900)
    m[:, :256] = float("-inf")
    m[:, 600:700] = torch.randn(2, 100)
    m[1, 768:] = float("-inf")
    plan, counts, tiles, stats, _ = worklist(case, mask=m)
    got = gpu_classes(plan, counts, tiles)
    want = oracle_classes(case, plan, mask=m)
    assert np.array_equal(got == 0, want == 0)
    # the all-zero tiles stay FULL, the mixed ones are PARTIAL
    assert got[0, 2] == 1 and got[0, 4] == 2 and got[0, 5] == 2
    # a tile with finite non-zero mask values is never FULL (that would drop its bias)
    assert want[0, 4] == 2 and want[0, 5] == 2
    assert np.all(want[got == 1] == 1)


LOG2E32 = np.float32(1.4426950408889634)


def check_gathered_lists(case, plan, ws, z, keep, units=None):
    """Top-k on the many-row path: each unit's gathered key list holds the
    keys some row of the unit keeps by the oracle's per-row sort -- first those
    every row of the unit keeps, then the others, each group in key order;
    each entry's rows [lo, hi) are exactly the unit's rows keeping that key;
    its bias is z_j * log2(e) (fp32); the last tile is padded with entries no
    row keeps; counts[item] is the number of 128-key tiles, and exactly the
    tiles made only of keys every row keeps are FULL in the work list."""
    p = case["params"]
    B, Sq, H, _ = case["q"].shape
    Sk = case["k"].shape[1]
    n_rt, nk, KT = plan["n_row_tiles"], plan["n_k_tiles"], plan["keys_per_tile"]
    n_items = plan["n_items"]
    w = ws.cpu()
    counts = w[plan["off_counts"]:plan["off_counts"] + 4 * n_items].view(torch.int32).numpy()
    tiles = w[plan["off_tiles"]:plan["off_tiles"] + 4 * n_items * nk].view(torch.int32).numpy().reshape(n_items, nk)
    lists = w[plan["off_topk_list"]:plan["off_topk_list"] + 8 * n_items * nk * KT].view(torch.int32).numpy()
    lists = lists.reshape(n_items, nk * KT, 2).view(np.uint32)
    keys = np.arange(Sk)
    for b in range(B):
        for h in range(H):
            zn = z[b, h].numpy()
            ok = O.allowed_pairs(np.arange(Sq), keys, Sq, Sk, causal=p["causal"])
            kept = np.zeros((Sq, Sk), bool)
            for rt in range(n_rt):
                if units is not None and (b, h, rt) not in units:
                    continue
                r0, r1 = rt * 128, min(rt * 128 + 127, Sq - 1)
                for i in range(r0, r1 + 1):
                    kept[i, O.topk_kept_row(zn, ok[i], keep)] = True
                item = (b * H + h) * n_rt + rt
                every = kept[r0:r1 + 1].all(axis=0)
                union = np.nonzero(kept[r0:r1 + 1].any(axis=0))[0]
                union = np.concatenate([union[every[union]], union[~every[union]]])
                n_every = int(every.sum())
                ent = lists[item, :counts[item] * KT]
                assert counts[item] == -(-len(union) // KT), (b, h, rt)
                want_tiles = [(t << 1) | int(t >= n_every // KT) for t in range(counts[item])]
                assert list(tiles[item, :counts[item]]) == want_tiles, (b, h, rt)
                real, pad = ent[:len(union)], ent[len(union):]
                assert np.array_equal(real[:, 0] & 0xffff, union), (b, h, rt)
                lo, hi = (real[:, 0] >> 16) & 0xff, real[:, 0] >> 24
                rows = kept[r0:r1 + 1, union]                  # [rows, keys]
                first = rows.argmax(axis=0)
                last = rows.shape[0] - 1 - rows[::-1].argmax(axis=0)
                assert np.array_equal(lo, first) and np.array_equal(hi, last + 1), (b, h, rt)
                assert all(rows[first[c]:last[c] + 1, c].all() for c in range(len(union))), "kept rows not an interval"
                bias = (zn[union].astype(np.float32) * LOG2E32).view(np.uint32)
                assert np.array_equal(real[:, 1], bias), (b, h, rt)
                assert np.all(((pad[:, 0] >> 16) & 0xff) == 128) and np.all((pad[:, 0] >> 24) == 0)


def test_topk_kept_sets_exact(golden):
    g = golden("fsa_mask_agreement.json")
    for seed, Sq, Sk, keep, causal, ties in [(0, 300, 300, 40, True, True), (1, 64, 500, 100, True, False),
                                             (2, 7, 260, 30, False, True), (3, 4, 4, 2, True, False),
                                             (4, 40, 9000, 3000, True, True),   # > 64 key buckets
                                             (5, 260, 700, 200, True, True),    # many rows over past keys
                                             (6, 200, 333, 50, False, True),    # many rows, not causal
                                             (7, 130, 2500, 3000, True, False),  # keep_window above every row
                                             (8, 300, 457, 120, True, True)]:    # key count not a multiple of 4
        case = W.random_case(seed, B=1, Sq=Sq, Sk=Sk, Hq=2, Hkv=2, d=64, causal=causal)
        z = W.random_zero_hold_states(seed, 1, 2, Sk, ties=ties)
        plan, counts, tiles, stats, ws = worklist(case, zero_hold_states=z, keep_window=keep)
        e = ws.cpu()[plan["off_topk_e"]:plan["off_topk_e"] + 4 * 2 * Sk].view(torch.int32).numpy()
        e = e.reshape(2, Sk).astype(np.int64)
        off = Sk - Sq
        n_match = n_total = 0
        for h in range(2):
            ok = O.allowed_pairs(np.arange(Sq), np.arange(Sk), Sq, Sk, causal=causal)
            for i in range(Sq):
                want = np.zeros(Sk, bool)
                want[O.topk_kept_row(z[0, h].numpy(), ok[i], keep)] = True
                got = ok[i] & (i < e[h])
                n_match += int((got == want).sum())
                n_total += Sk
        assert n_match / n_total == g["position_match"]
        if plan["path"] == fa._lib.FA_PATH_PREFILL:
            check_gathered_lists(case, dict(plan), ws, z, keep)
        else:
            # EMPTY tiles are a subset of the truly empty ones, and no kept pair is lost
            got = gpu_classes(plan, counts, tiles)
            want = oracle_classes(case, plan, zero_hold_states=z, keep_window=keep)
            assert np.all(want[got == 0] == 0)


def test_inconsistent_lengths_are_reported():
    """A sequence longer than the max_seqlen the plan was sized for is caught on
    the device (no out-of-range access): its item is skipped and the error word
    says FA_ERR_DEVICE_BOUNDS."""
    q, k, v, cu_q, cu_k = W.random_varlen(3, 2, 2, 300, 4, 2, 64, min_q=1, min_k=1)
    lk = int((cu_k[1:] - cu_k[:-1]).max())
    p = W.base_params(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=2, max_seqlen_k=max(1, lk - 1),
                      causal=True)
    out, lse, ws = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), **to_dev(p))
    rc, info = fa.fa_check_device_error(ws)
    assert rc == fa._lib.FA_ERR_DEVICE_BOUNDS


def test_topk_kept_sets_at_full_workload_shape():
    """Kept sets of the dynamic top-k workload itself (B=2, H=16, T=8192,
    keep_window=2048, causal), with ties quantised in: the expiry rows the
    GPU writes, read back as per-row kept sets, equal the oracle's per-row
    sort on sampled rows of every (b, h), including the rows where the
    window first fills (2047, 2048) and the last row
    (flash-sparse-attention issue 11, "Current Status": position match 1.0)."""
    case = W.dynamic_topk(seed=0)
    p = dict(case["params"])
    B, Sq, H, _ = case["q"].shape
    Sk = case["k"].shape[1]
    keep = p["keep_window"]
    z = torch.round(p["zero_hold_states"] * 4.0) / 4.0   # ties on
    plan, counts, tiles, stats, ws = worklist(case, zero_hold_states=z)
    e = ws.cpu()[plan["off_topk_e"]:plan["off_topk_e"] + 4 * B * H * Sk].view(torch.int32).numpy()
    e = e.reshape(B, H, Sk).astype(np.int64)
    off = Sk - Sq
    rng = np.random.default_rng(5)
    keys = np.arange(Sk)
    for b in range(B):
        for h in range(H):
            zn = z[b, h].numpy()
            rows = {0, keep - 2, keep - 1, keep, keep + 1, Sq - 1} | set(rng.integers(0, Sq, 6).tolist())
            for i in sorted(rows):
                cand = O.allowed_pairs([i], keys, Sq, Sk, causal=True)[0]
                want = np.zeros(Sk, bool)
                want[O.topk_kept_row(zn, cand, keep)] = True
                got = (keys <= i + off) & (i < e[b, h])
                assert np.array_equal(got, want), (b, h, i, int((got != want).sum()))
    # the gathered lists of units where the window is filling, just full, and at the end
    units = {(0, 0, 0), (0, 3, 15), (0, 5, 16), (1, 7, 17), (1, 15, 63), (0, 9, 40)}
    check_gathered_lists(case, dict(plan), ws, z, keep, units=units)


@pytest.mark.parametrize("seed,B,Sq,Sk,Hq,Hkv,d,extra", [
    (0, 2, 300, 700, 4, 2, 128, dict(causal=True)),                                   # past KV, ragged
    (1, 1, 260, 520, 2, 2, 64, dict(causal=True, window_left=150, window_right=20)),  # window
    (2, 1, 400, 200, 2, 1, 128, dict(causal=True)),                                   # q_len > kv_len
    (3, 1, 200, 333, 2, 2, 64, dict(causal=False)),
])
def test_prefill_inline_schedule_counts(seed, B, Sq, Sk, Hq, Hkv, d, extra):
    """Without a mask the prefill kernel classifies its own tiles (no
    scheduler kernel runs): the counters it writes equal the FULL / PARTIAL /
    EMPTY classes recomputed from the oracle's logits, and EMPTY tiles are
    never among the scheduled ones (their count is exact)."""
    case = W.random_case(seed, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, d=d, **extra)
    rc, plan = fa.fa_fwd_plan(case["q"], case["k"], case["v"], **case["params"])
    assert rc == 0 and plan["path"] == fa._lib.FA_PATH_PREFILL and plan["n_kernels"] == 1
    ws = fa.alloc_workspace(plan["workspace_bytes"], DEV)
    ws[plan["off_stats"]:plan["off_stats"] + 24] = 7          # stale counters must be overwritten
    run_gpu(case, workspace=ws)
    stats = ws.cpu()[plan["off_stats"]:plan["off_stats"] + 24].view(torch.int64).numpy()
    want = oracle_classes(case, plan)
    n_kt_seq = -(-Sk // plan["keys_per_tile"])
    if Sk % plan["keys_per_tile"]:
        # a tile reaching past the last key is never FULL: the kernel masks the
        # keys it lacks (the scheduler kernel applies the same rule)
        last = want[:, n_kt_seq - 1]
        last[last == 1] = 2
    assert stats[0] == int((want == 1).sum())
    assert stats[1] == int((want == 2).sum())
    assert stats[2] == int((want[:, :n_kt_seq] == 0).sum())
