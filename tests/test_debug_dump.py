"""The prefill kernel's debug dump against the fp64 oracle's intermediate
values: for one (sequence, head, query tile), the raw scores S of every key
tile in the unit's list equal Q K^T, and P equals exp2(logit x log2 e - ref)
rounded to the input type where the pair rules keep the key, 0 elsewhere
(flash-sparse-attention issue 11 "Next Steps": dump one block's logits, mask
and output for step-by-step comparison).  The outputs match the oracle as
fa_fwd's do.  The checker itself is tested on the CPU with dumps built from
the definitions, and with planted mistakes that it must reject."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as O
from parity_util import DEV, compare, run_oracle, to_dev


def check_dump(c, seq, head, rt, tiles, S, P, R):
    """Assert that a dump (S, P, ref per key-tile entry) is the unit's."""
    p = c["params"]
    G = c["q"].shape[2] // c["k"].shape[2]
    Sq, Sk = c["q"].shape[1], c["k"].shape[1]
    rows = np.arange(rt * 128, rt * 128 + 128)
    live = rows < Sq
    qr = c["q"][seq, rows[live], head].double().numpy()
    kk = c["k"][seq, :, head // G].double().numpy()
    scale = p["scale"] or 1.0 / math.sqrt(c["q"].shape[3])
    x = O.logits_rows(qr, kk, rows[live], Sq, Sk, scale=scale, causal=p["causal"], window_left=p["window_left"],
                      window_right=p["window_right"], softcap=p["softcap"])
    for it, ent in enumerate(tiles):
        kt = int(ent) >> 1
        cols = np.arange(kt * 128, kt * 128 + 128)
        inb = cols < Sk
        want_s = qr @ kk[cols[inb]].T
        got_s = S[it][live][:, inb]
        assert np.abs(got_s - want_s).max() <= 1e-3 * max(1.0, np.abs(want_s).max()), f"S of entry {it}"
        logit = np.full((int(live.sum()), 128), -np.inf)
        logit[:, inb] = x[:, cols[inb]]
        fin = np.isfinite(logit)
        got_p = P[it][live]
        assert (got_p[~fin] == 0).all(), f"P of dropped keys, entry {it}"
        want_p = np.exp2(logit * math.log2(math.e) - R[it][live][:, None])
        assert np.allclose(got_p[fin], want_p[fin], rtol=2e-2, atol=1e-6), f"P of entry {it}"


def _definition_dump(c, seq, head, rt):
    """A dump built from the definitions (the reference is the row maximum
    over the tile's kept logits, P rounded to bf16), and its tile list."""
    p = c["params"]
    G = c["q"].shape[2] // c["k"].shape[2]
    Sq, Sk = c["q"].shape[1], c["k"].shape[1]
    rows = np.arange(rt * 128, rt * 128 + 128)
    qr = np.zeros((128, c["q"].shape[3]))
    live = rows < Sq
    qr[live] = c["q"][seq, rows[live], head].double().numpy()
    kk = c["k"][seq, :, head // G].double().numpy()
    x = O.logits_rows(qr, kk, rows, Sq, Sk, scale=p["scale"], causal=p["causal"], window_left=p["window_left"],
                      window_right=p["window_right"], softcap=p["softcap"])
    x[~live] = -np.inf
    n_kt = -(-Sk // 128)
    tiles, S, P, R = [], [], [], []
    for kt in range(n_kt):
        cols = np.arange(kt * 128, min(kt * 128 + 128, Sk))
        blk = x[:, cols] * math.log2(math.e)
        if not np.isfinite(blk).any():
            continue
        tiles.append(kt << 1)
        s = np.zeros((128, 128))
        s[:, :len(cols)] = qr @ kk[cols].T
        ref = np.where(np.isfinite(blk).any(axis=1), np.max(np.where(np.isfinite(blk), blk, -1e300), axis=1), 0.0)
        pp = np.zeros((128, 128))
        pp[:, :len(cols)] = np.exp2(blk - ref[:, None])
        pp = torch.from_numpy(pp).to(torch.bfloat16).double().numpy()
        S.append(s); P.append(pp); R.append(ref)
    return tiles, np.array(S), np.array(P), np.array(R)


@pytest.mark.parametrize("extra", [dict(causal=True), dict(causal=True, window_left=150, softcap=20.0)])
def test_checker_accepts_the_definition_and_rejects_mistakes(extra):
    c = W.random_case(1710, B=1, Sq=300, Sk=520, Hq=2, Hkv=1, d=64, **extra)
    c["params"]["scale"] = 0.125
    tiles, S, P, R = _definition_dump(c, 0, 1, 2)
    check_dump(c, 0, 1, 2, tiles, S, P, R)
    with pytest.raises(AssertionError):   # S of the wrong keys (transposed tile order)
        check_dump(c, 0, 1, 2, tiles, S[::-1], P, R)
    with pytest.raises(AssertionError):   # P against a reference off by one
        check_dump(c, 0, 1, 2, tiles, S, P, R + 1.0)
    P2 = P.copy()
    P2[0][:, 127] = 0.5                   # a value where the last column is dropped or differs
    with pytest.raises(AssertionError):
        check_dump(c, 0, 1, 2, tiles, S, P2, R)


@pytest.mark.gpu
@pytest.mark.parametrize("seq,head,rt,extra", [
    (0, 1, 1, dict(causal=True)),
    (1, 3, 2, dict(causal=True, window_left=150, softcap=20.0)),
])
def test_debug_dump(seq, head, rt, extra):
    import masked_flash_attention_gb300 as fa
    c = W.random_case(1700 + seq, B=2, Sq=300, Sk=520, Hq=4, Hkv=2, d=128, **extra)
    p = c["params"]
    out, lse, ws, dump = fa.fa_fwd_debug_dump(c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV), seq, head, rt,
                                              **to_dev(p))
    torch.cuda.synchronize()
    rc, info = fa.fa_check_device_error(ws)
    assert rc == 0, (rc, info)
    ref_o, ref_l = run_oracle(c)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "debug dump call")
    _, plan = fa.fa_fwd_plan(c["q"], c["k"], c["v"], **p)
    item = (seq * plan["n_heads_sched"] + head) * plan["n_row_tiles"] + rt
    w = ws.cpu().numpy().view(np.uint8)
    oc, ot, nk = plan["off_counts"], plan["off_tiles"], plan["n_k_tiles"]
    count = int(w[oc + 4 * item:oc + 4 * item + 4].view(np.int32)[0])
    tiles = w[ot + 4 * item * nk:ot + 4 * (item * nk + count)].view(np.int32)
    assert count > 0
    check_dump(c, seq, head, rt, tiles, dump["S"].cpu().numpy()[:count], dump["P"].cpu().numpy()[:count],
               dump["ref"].cpu().numpy()[:count])
