"""Benchmark of the masked flash-attention forward on GB300.

One step = one fa_fwd call over one batch of the workload (all of the hot
path: top-k preparation or mask summary when the workload has one, tile
classification, the attention kernel and the split combine).

Default workload: causal prefill over past KV with grouped-query heads
(B=4, Hq=32, Hkv=8, d=128, 512 new queries over 4096 keys), metric "useful
TFLOP/s": 4*d FLOP per (query, key) pair that the mask keeps, per query head.
``--workload paged_varlen_decode`` reports KV-cache GB/s (K/V bytes inside
each sequence's window) instead; ``--workload paged_decode_append`` serves the
same batch through fa_fwd_kvcache (cached keys plus each sequence's new token
read from its own tensor, and appended to the cache), reporting the same bytes
plus the appended rows.

Rules kept here: W >= 3 untimed warm-up steps; each timed step is bracketed by
CUDA events on the launching stream; between timed steps L2 is flushed by
writing a 256 MB buffer and then reading another (outside the events: the
read evicts the write's dirty lines, whose write-back would otherwise fall
inside the timed kernel), except where a step reads
several times more than L2 holds (the decode workloads: 749 MB of K/V per
step), which the rules allow instead of a flush: there the flush's dirty lines
would be written back during the timed kernel; inputs are resident in HBM when
a step starts.  ``e2e`` repeats the measurement through the same public call
with the inputs copied from pinned host memory and the outputs copied back
inside the timed region.  Under torchrun every rank runs its own batch
(independent problems, no collective on the data path): weak scaling.

``--impl reference`` times the fp64 CPU oracle (the method's plain
definition) on the host cores instead, on a bounded sample of the same
workload, and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "masked attn fwd useful TFLOP/s (prefill) and KV-cache GB/s (decode), 1×GB300"
METRIC_BWD = "masked attn bwd useful TFLOP/s (dq, dk, dv: 10 d FLOP per kept pair), 1×GB300"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300 L2
# a step that reads at least this much needs no flush: its own reads evict
# whatever the previous step left in L2 before they could reuse it
NO_FLUSH_READ_BYTES = 4 * L2_BYTES


def flushes_l2(units, bwd=False):
    """True when timed steps are separated by an L2 flush: unless a step reads
    at least NO_FLUSH_READ_BYTES (known only for the byte-bound workloads;
    the backward always flushes)."""
    return bwd or units["bytes"] is None or units["bytes"] < NO_FLUSH_READ_BYTES
CSRC = os.path.join(ROOT, "masked_flash_attention_gb300", "csrc")
KERNEL_SOURCES = {"prefill_kernel": ["prefill_sm103.cu", "tc_sm103.cuh", "fa_device.cuh"],
                  "decode_kernel": ["decode.cu", "mma_sync.cuh", "fa_device.cuh"]}
# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum; see profiles/), keyed
# by workload and kernel, with the hash of the kernel's sources at capture
# time (comments and white space left out): once the kernel's code changes the
# figure no longer applies and is reported as null.
MEASURED_TRAFFIC = {
    ("causal_prefill_past_kv", "prefill_kernel"): ("701a81111927638c", 103775488 + 11407872),
    ("gpt2_small_layer", "prefill_kernel"): ("701a81111927638c", 37847040 + 120832),
    ("llama3_8b_layer", "prefill_kernel"): ("701a81111927638c", 100772096 + 37414656),
    ("dynamic_topk", "prefill_kernel"): ("701a81111927638c", 201289216 + 52963584),
    ("paged_varlen_decode", "decode_kernel"): ("41c2ad86020fef38", 752926208 + 9257472),
    ("paged_decode_append", "decode_kernel"): ("41c2ad86020fef38", 752866560 + 9434368),
}


def code_text(src):
    """A C++/CUDA source without its comments and with runs of white space
    collapsed: what the compiler sees, so that editing a comment does not
    mark a measurement stale."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_hash(kernel):
    import hashlib
    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            m.update(code_text(fh.read()).encode())
    return m.hexdigest()[:16]


def measured_traffic(workload, kernel):
    rec = MEASURED_TRAFFIC.get((workload, kernel))
    if rec is None or rec[0] != kernel_hash(kernel):
        return None
    return rec[1]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"],
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# Algorithmic work (counted from the definition, not from the kernels)
# ---------------------------------------------------------------------------

def useful_pairs(case):
    """Number of (query row, key, q-head) triples the mask keeps, counted with
    closed forms for the causal/window rules and exactly for top-k."""
    p = case["params"]
    q, k = case["q"], case["k"]
    if p["cu_seqlens_q"] is not None:
        cu_q = p["cu_seqlens_q"].tolist()
        cu_k = p["cu_seqlens_k"].tolist()
        lens = [(cu_q[i + 1] - cu_q[i], cu_k[i + 1] - cu_k[i]) for i in range(len(cu_q) - 1)]
        Hq = q.shape[1]
    else:
        lens = [(q.shape[1], k.shape[1])] * q.shape[0]
        Hq = q.shape[2]
    total = 0
    for Sq, Sk in lens:
        off = Sk - Sq
        i = np.arange(Sq, dtype=np.int64)
        hi = np.full(Sq, Sk - 1, dtype=np.int64)
        lo = np.zeros(Sq, dtype=np.int64)
        if p["causal"]:
            hi = np.minimum(hi, i + off)
        if p["window_left"] >= 0:
            lo = np.maximum(lo, i + off - p["window_left"])
        if p["window_right"] >= 0:
            hi = np.minimum(hi, i + off + p["window_right"])
        cnt = np.maximum(hi - lo + 1, 0)
        if p["zero_hold_states"] is not None:
            cnt = np.minimum(cnt, p["keep_window"])
        total += int(cnt.sum()) * Hq
    if p["mask"] is not None:  # dense mask: its finite entries among the allowed pairs
        fin = torch.isfinite(p["mask"]).numpy()
        if fin.ndim == 2:
            fin = fin[None, None]
        total = 0
        for b, (Sq, Sk) in enumerate(lens):
            i = np.arange(Sq, dtype=np.int64)[:, None]
            j = np.arange(Sk, dtype=np.int64)[None, :]
            off = Sk - Sq
            ok = np.ones((Sq, Sk), dtype=bool)
            if p["causal"]:
                ok &= j <= i + off
            if p["window_left"] >= 0:
                ok &= j >= i + off - p["window_left"]
            if p["window_right"] >= 0:
                ok &= j <= i + off + p["window_right"]
            for h in range(Hq):
                mb = fin[b if fin.shape[0] > 1 else 0, h if fin.shape[1] > 1 else 0, :Sq, :Sk]
                total += int((mb & ok).sum())
    return total


def kv_window_bytes(case):
    """K and V bytes inside each sequence's window (decode workloads)."""
    p = case["params"]
    cu_k = p["cu_seqlens_k"].tolist()
    cu_q = p["cu_seqlens_q"].tolist()
    Hkv, d = case["k"].shape[-2], case["k"].shape[-1]
    tot = 0
    for s in range(len(cu_k) - 1):
        Sk, Sq = cu_k[s + 1] - cu_k[s], cu_q[s + 1] - cu_q[s]
        lo = max(0, (Sk - Sq) - p["window_left"]) if p["window_left"] >= 0 else 0
        tot += (Sk - lo) * Hkv * d * 2 * 2
    return tot


def algorithmic_io_bytes(case):
    """Compulsory HBM bytes of one forward: Q, K, V read once, O and LSE written."""
    q, k, v = case["q"], case["k"], case["v"]
    lse = q.numel() // q.shape[-1] * 4
    return (q.numel() + k.numel() + v.numel() + q.numel()) * 2 + lse


def _as_dtype(case, dtype):
    """The workload with q, k, v in the requested input type (for "f16" the
    bf16 draws converted to fp16)."""
    if dtype == "bf16":
        return case
    t = torch.float16
    out = dict(case, name=case["name"] + "_f16", q=case["q"].to(t), k=case["k"].to(t), v=case["v"].to(t))
    if "kvcache" in case:
        out["kvcache"] = dict(case["kvcache"], k_new=case["kvcache"]["k_new"].to(t),
                              v_new=case["kvcache"]["v_new"].to(t))
    return out


def workload_units(case, name):
    d = case["q"].shape[-1]
    if name in ("paged_varlen_decode", "paged_decode_append"):
        b = kv_window_bytes(case)
        if "kvcache" in case:  # the append writes the active K and V rows
            b += 2 * case["kvcache"]["k_new"].numel() * case["kvcache"]["k_new"].element_size()
        return dict(metric_units=b / 1e9, unit="GB/s", bound="hbm",
                    flops=4.0 * d * useful_pairs(case), bytes=b)
    f = 4.0 * d * useful_pairs(case)
    return dict(metric_units=f / 1e12, unit="TFLOP/s", bound="tensor", flops=f, bytes=None)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _dist():
    """torch.distributed when launched with WORLD_SIZE > 1: NCCL between GPUs,
    gloo on a host without one (where the multi-rank host logic is tested)."""
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist
    return None


def max_over_ranks(dist, x, device="cpu"):
    """The slowest rank's figure: each rank times its own replica."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_case(args, rank):
    """Rank ``rank``'s replica: the workload's shapes drawn from its own seed.
    Ranks share no data, so the step needs no collective."""
    return _as_dtype(W.WORKLOADS[args.workload](seed=args.seed + rank), args.dtype)


def job_value(metric_units, world, ms_per_step):
    """Whole-job throughput: each of ``world`` ranks runs one replica per step."""
    return metric_units * world / (ms_per_step / 1e3)


def run_gpu(args):
    import masked_flash_attention_gb300 as fa

    dist = _dist()
    rank = dist.get_rank() if dist else 0
    world = dist.get_world_size() if dist else 1
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = replica_case(args, rank)
    units = workload_units(case, args.workload)
    bwd = args.pass_ == "bwd"
    if bwd:
        # useful backward work: 5 products of 2 d FLOP per kept pair (S, dP,
        # dV, dK, dQ) = 2.5 x the forward's 4 d
        assert units["bound"] == "tensor" and "kvcache" not in case, "--pass bwd takes the prefill workloads"
        units = dict(units, flops=units["flops"] * 2.5, metric_units=units["metric_units"] * 2.5)
    p = dict(case["params"])
    gp = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    q, k, v = case["q"].to(dev), case["k"].to(dev), case["v"].to(dev)
    stream = torch.cuda.current_stream()
    # the two-source form (cached keys + the step's active rows, appended)
    kvx = {kk: (vv.to(dev) if isinstance(vv, torch.Tensor) else vv) for kk, vv in case["kvcache"].items()} \
        if "kvcache" in case else None

    def call(q_, k_, v_, kvx_, **kw):
        if kvx_ is None:
            return fa.fa_fwd(q_, k_, v_, **kw, **gp)
        return fa.fa_fwd_kvcache(q_, k_, v_, kvx_["k_new"], kvx_["v_new"], kvx_["cache_seqlens"],
                                 append=kvx_["append"], **kw, **gp)

    if kvx is None:
        rc, plan = fa.fa_fwd_plan(q, k, v, stream=stream.cuda_stream, **gp)
    else:
        rc, plan = fa.fa_fwd_kvcache_plan(q, k, v, kvx["k_new"], kvx["v_new"], kvx["cache_seqlens"],
                                          append=kvx["append"], stream=stream.cuda_stream, **gp)
    assert rc == 0, rc
    ws = fa.alloc_workspace(plan["workspace_bytes"], dev)
    out = torch.empty_like(q)
    lse_shape = (q.shape[1], q.shape[0]) if p["cu_seqlens_q"] is not None else (q.shape[0], q.shape[2], q.shape[1])
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    big_reads = not flushes_l2(units, bwd)

    def flush_l2():
        # the write evicts the inputs; the read of another buffer then evicts
        # the write's dirty lines, so that their write-back to HBM happens
        # here and not inside the timed kernel
        if not big_reads:
            flush.zero_()
            flush_rd.max()
    ev_kb = torch.cuda.Event(enable_timing=True)
    ev_ke = torch.cuda.Event(enable_timing=True)
    ev_kb.record(); ev_ke.record()

    def step(timing=False, kb=None, ke=None, ka=None):
        call(q, k, v, kvx, out=out, lse=lse, workspace=ws, stream=stream.cuda_stream, event_begin=kb,
             event_end=ke, event_attn_end=ka)

    if bwd:
        # the forward once (untimed) for out and lse; each step is one fa_bwd
        step()
        gd = torch.Generator().manual_seed(args.seed + 7)
        hdout = torch.randn(case["q"].shape, generator=gd, dtype=torch.float32).to(case["q"].dtype)
        dout = hdout.to(dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc, plan = fa.fa_bwd_plan(q, k, v, out, lse, dout, stream=stream.cuda_stream, **gp)
        assert rc == 0, rc
        ws = fa.alloc_workspace(plan["workspace_bytes"], dev)

        def step(timing=False, kb=None, ke=None, ka=None):  # noqa: F811
            fa.fa_bwd(q, k, v, out, lse, dout, dq=gq, dk=gk, dv=gv, workspace=ws, stream=stream.cuda_stream,
                      event_begin=kb, event_end=ke, **gp)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    rc_, info = fa.fa_check_device_error(ws)
    assert rc_ == 0, (rc_, info)

    # ---- device-resident timing ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    # per step: the attention kernel's begin, the end of the attention kernel
    # itself, the end of the call's last pass (the decode path's split
    # combine).  A prefill call has no pass after its kernel: its steps record
    # no third event, as each timing event on the stream costs about 2 us of
    # the step.
    after_pass = bwd or plan["path"] == fa._lib.FA_PATH_DECODE
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        # one more untimed step: the sampler's start-up pause leaves the GPU
        # idle, and the first step after an idle GPU runs slow
        flush_l2()
        step()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            kev[i][0].record(); kev[i][1].record(); kev[i][2].record()  # materialise the handles
            ev[i][0].record()
            step(kb=kev[i][0], ke=kev[i][2] if after_pass else None, ka=None if bwd else kev[i][1])
            ev[i][1].record()
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # the dominant kernel alone (the backward: its three kernels); the passes
    # after it (split combine) are reported beside it
    kern_ms = [a.elapsed_time(c if bwd else b) for a, b, c in kev]
    after_ms = [b.elapsed_time(c) if after_pass and not bwd else 0.0 for a, b, c in kev]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, dev)
    if dist:
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = job_value(units["metric_units"], world, ms_per_step)

    # ---- end to end: pinned host inputs in, outputs back, same public call ----
    # Pipelined over two buffer sets, as a serving loop would run: step i's
    # inputs are copied in (copy-in stream) while step i - 1 computes, and its
    # outputs copied out (copy-out stream) while step i + 1 computes.  Every
    # copy of every step is inside the timed region.
    hq, hk, hv = (case["q"].pin_memory(), case["k"].pin_memory(), case["v"].pin_memory())
    hx = {kk: vv.pin_memory() for kk, vv in case["kvcache"].items() if isinstance(vv, torch.Tensor)} \
        if kvx is not None else {}
    if not bwd:
        h_in = [hq, hk, hv, *hx.values()]
        sets = []
        for _ in range(2):
            d_in = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
            dx_ = dict(kvx, **{kk: torch.empty_like(kvx[kk]) for kk in hx}) if kvx is not None else None
            d_in += [dx_[kk] for kk in hx]
            d_out = [torch.empty_like(out), torch.empty_like(lse)]
            sets.append(dict(d_in=d_in, dx=dx_, d_out=d_out,
                             h_out=[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out]))

        def compute(st_, s_):
            dq_, dk_, dv_ = st_["d_in"][:3]
            call(dq_, dk_, dv_, st_["dx"], out=st_["d_out"][0], lse=st_["d_out"][1], workspace=ws,
                 stream=s_.cuda_stream)
    else:
        # inputs q, k, v, out, lse, dout in; dq, dk, dv back
        h_in = [hq, hk, hv, out.cpu().pin_memory(), lse.cpu().pin_memory(), hdout.pin_memory()]
        sets = []
        for _ in range(2):
            d_in = [torch.empty_like(t) for t in (q, k, v, out, lse, dout)]
            d_out = [torch.empty_like(t) for t in (gq, gk, gv)]
            sets.append(dict(d_in=d_in, d_out=d_out,
                             h_out=[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out]))

        def compute(st_, s_):  # noqa: F811
            qq, kk_, vv, oo, ll, dd = st_["d_in"]
            g1, g2, g3 = st_["d_out"]
            fa.fa_bwd(qq, kk_, vv, oo, ll, dd, dq=g1, dk=g2, dv=g3, workspace=ws, stream=s_.cuda_stream, **gp)
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["d_out"])
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]   # a set's inputs landed
    ev_cmp = [torch.cuda.Event() for _ in range(2)]  # a set's computation done
    ev_out = [torch.cuda.Event() for _ in range(2)]  # a set's outputs copied out

    def run_steps(n):
        for i in range(n):
            b = i & 1
            st_ = sets[b]
            s_in.wait_event(ev_cmp[b])  # the computation two steps back has read these inputs
            with torch.cuda.stream(s_in):
                for d_, h_ in zip(st_["d_in"], h_in):
                    d_.copy_(h_, non_blocking=True)
            ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])  # these outputs of two steps back have left
            with torch.cuda.stream(s_cmp):
                compute(st_, s_cmp)
            ev_cmp[b].record(s_cmp)
            s_out.wait_event(ev_cmp[b])
            with torch.cuda.stream(s_out):
                for h_, d_ in zip(st_["h_out"], st_["d_out"]):
                    h_.copy_(d_, non_blocking=True)
            ev_out[b].record(s_out)

    torch.cuda.synchronize()
    run_steps(max(2, args.warmup))
    torch.cuda.synchronize()
    e2e_a, e2e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_a.record(s_in)
    run_steps(args.steps)
    e2e_b.record(s_out)  # after the last copy out, which follows every computation
    torch.cuda.synchronize()
    e2e_ms = [e2e_a.elapsed_time(e2e_b)]
    e2e_total = sum(e2e_ms)
    e2e_total = max_over_ranks(dist, e2e_total, dev)
    e2e_value = job_value(units["metric_units"], world, e2e_total / args.steps)
    rc_, info = fa.fa_check_device_error(ws)
    assert rc_ == 0, (rc_, info)
    # the scheduler's counters of the last call: key tiles computed FULL or
    # PARTIAL, and left out as EMPTY (never computed)
    st = ws[plan["off_stats"]:plan["off_stats"] + 24].cpu().view(torch.int64).tolist() if not bwd else None

    if rank != 0:
        return None
    pk = peaks()
    kern_avg = sum(kern_ms) / len(kern_ms)
    if units["bound"] == "tensor":
        achieved = units["flops"] / (kern_avg / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16"], 4)}
    else:
        achieved = units["bytes"] / (kern_avg / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4)}
    roof["peak_source"] = pk["src"]
    roof["kernel"] = "decode_kernel" if plan["path"] == fa._lib.FA_PATH_DECODE else "prefill_kernel"
    if bwd:
        roof["kernel"] = "backward (delta_kernel, dkdv_kernel, dq_kernel)"
    roof["kernel_ms"] = round(kern_avg, 5)
    if not bwd:
        roof["after_kernel_ms"] = round(sum(after_ms) / len(after_ms), 5)  # split combine (decode), else ~0
    roof["traffic"] = args.traffic if args.traffic is not None else measured_traffic(args.workload, roof["kernel"])
    if units["bytes"] is not None or roof["bound"] == "tensor":
        roof["algorithmic_bytes"] = units["bytes"] if units["bytes"] is not None else algorithmic_io_bytes(case)
    line = {
        "metric": METRIC if args.pass_ == "fwd" else METRIC_BWD,
        "value": round(value, 3),
        "unit": units["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": args.dtype,
        "data": "synthetic",
        "config": {"workload": case["name"], "seed": args.seed, "pass": args.pass_,
                   "l2": (f"no flush: each step reads {units['bytes'] / 1e6:.0f} MB, more than 4x the {L2_BYTES >> 20} MB L2"
                          if big_reads else "flushed between timed steps (256 MB write, then a 256 MB read so "
                          "that no dirty line is left, outside the events)"),
                   "parallelism": f"replica per GPU x{world}", "path": plan["path"],
                   "n_items": plan["n_items"], "n_splits": plan["n_splits"]},
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 3), "unit": units["unit"], "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_total / args.steps, 5),
                "overlap": "two buffer sets: a step's copies in and out overlap its neighbours' computation",
                "l2": "each step's inputs arrive by its own host-to-device copies"},
        "gpu_launches": int(plan["n_kernels"]) * args.steps,
        "latency_us": round(ms_per_step * 1e3, 2),
        "clocks": clk.summary(),
    }
    if st is not None:
        line["sched"] = {"full": st[0], "partial": st[1], "empty": st[2]}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, units, args)
    return line


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def _oracle_sample(case, n_heads):
    """Oracle on the first ``n_heads`` (sequence, head) pairs of the workload;
    returns (seconds, fraction of the workload's units covered)."""
    from oracle import attention as O
    p = case["params"]
    q, k, v = case["q"], case["k"], case["v"]
    packed = p["cu_seqlens_q"] is not None
    Hq = q.shape[-2]
    Hkv = k.shape[-2]
    G = Hq // Hkv
    pairs = [(b, h) for b in range(len(p["cu_seqlens_q"]) - 1 if packed else q.shape[0])
             for h in range(Hq)]
    sel = pairs[:n_heads]
    qn = q.float().numpy(); kn = k.float().numpy(); vn = v.float().numpy()
    t0 = time.perf_counter()
    for b, h in sel:
        if packed:
            cu_q = p["cu_seqlens_q"].tolist(); cu_k = p["cu_seqlens_k"].tolist()
            Sk = cu_k[b + 1] - cu_k[b]
            qb = qn[cu_q[b]:cu_q[b + 1], h]
            if p["block_table"] is not None:
                kb = O.gather_paged(kn, p["block_table"][b].numpy(), Sk)[:, h // G]
                vb = O.gather_paged(vn, p["block_table"][b].numpy(), Sk)[:, h // G]
            else:
                kb = kn[cu_k[b]:cu_k[b + 1], h // G]; vb = vn[cu_k[b]:cu_k[b + 1], h // G]
        else:
            qb = qn[b, :, h]; kb = kn[b, :, h // G]; vb = vn[b, :, h // G]
            Sk = kb.shape[0]
        z = None if p["zero_hold_states"] is None else p["zero_hold_states"][b, h].numpy()
        m = None if p["mask"] is None else p["mask"].numpy()
        O.attention_rows(qb, kb, vb, np.arange(qb.shape[0]), qb.shape[0], Sk,
                         scale=p["scale"], causal=p["causal"], window_left=p["window_left"],
                         window_right=p["window_right"], softcap=p["softcap"], mask_rows=m, z=z,
                         keep_window=p["keep_window"])
    dt = time.perf_counter() - t0
    return dt, len(sel) / len(pairs)


def _n_pairs(case, n):
    p = case["params"]
    total = (len(p["cu_seqlens_q"]) - 1 if p["cu_seqlens_q"] is not None else case["q"].shape[0]) * \
        case["q"].shape[-2]
    return min(n, total)


def _pick_heads(case, budget_s):
    """Number of (sequence, head) pairs whose oracle run takes about budget_s."""
    dt1, _ = _oracle_sample(case, 1)
    return max(1, int(budget_s / max(dt1, 1e-3))), dt1


def _oracle_bwd_sample(case):
    """Backward oracle on the first K/V head's q-head group of the first
    sequence; returns (seconds, fraction of the workload's units covered)."""
    from oracle import backward as B
    p = dict(case["params"])
    q, k, v = case["q"], case["k"], case["v"]
    assert p["cu_seqlens_q"] is None, "fixed-length workloads"
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    g = torch.Generator().manual_seed(11)
    do = torch.randn(1, q.shape[1], G, q.shape[3], generator=g).to(q.dtype)
    t0 = time.perf_counter()
    B.attention_grad(q[:1, :, :G], k[:1, :, :1], v[:1, :, :1], do, **p)
    return time.perf_counter() - t0, G / (q.shape[0] * Hq)


def cpu_baseline(case, units, args, budget_s=None):
    budget_s = args.cpu_budget if budget_s is None else budget_s
    if getattr(args, "pass_", "fwd") == "bwd":
        dt, frac = _oracle_bwd_sample(case)
        return {"value": round(units["metric_units"] * frac / dt, 6), "unit": units["unit"],
                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                "sample": f"fp64 numpy backward oracle on one K/V head's q-head group of one sequence "
                          f"({frac * 100:.2f}% of the units) in {dt:.2f} s"}
    n, _ = _pick_heads(case, budget_s)
    dt, frac = _oracle_sample(case, n)
    val = units["metric_units"] * frac / dt
    n = _n_pairs(case, n)
    return {"value": round(val, 6), "unit": units["unit"], "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle on {n} of the workload's (sequence, q-head) pairs "
                      f"({frac * 100:.2f}% of the units) in {dt:.2f} s; numpy BLAS on all cores, "
                      "elementwise work single-threaded"}


def run_reference(args):
    dist_rank = int(os.environ.get("RANK", "0"))
    if dist_rank != 0:
        return None
    case = _as_dtype(W.WORKLOADS[args.workload](seed=args.seed), args.dtype)
    units = workload_units(case, args.workload)
    if args.pass_ == "bwd":
        units = dict(units, flops=units["flops"] * 2.5, metric_units=units["metric_units"] * 2.5)
        sample_fn = lambda: _oracle_bwd_sample(case)  # noqa: E731
        what = "fp64 numpy backward oracle on one K/V head's q-head group of one sequence"
    else:
        per_step_budget = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
        n, _ = _pick_heads(case, per_step_budget)
        sample_fn = lambda: _oracle_sample(case, n)  # noqa: E731
        what = f"fp64 numpy oracle on {_n_pairs(case, n)} (sequence, q-head) pairs"
    for _ in range(args.warmup):
        sample_fn()
    times, frac = [], 0.0
    for _ in range(args.steps):
        dt, frac = sample_fn()
        times.append(dt)
    ms = sum(times) / len(times) * 1e3
    val = units["metric_units"] * frac / (ms / 1e3)
    cores = len(os.sched_getaffinity(0))
    sample = (f"each step: {what} = {frac * 100:.2f}% of the workload; value scaled to the workload's units")
    return {
        "impl": "reference", "metric": METRIC if args.pass_ == "fwd" else METRIC_BWD, "value": round(val, 6), "unit": units["unit"],
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case["name"], "seed": args.seed, "pass": args.pass_},
        "cpu_baseline": {"value": round(val, 6), "unit": units["unit"], "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 6), "unit": units["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="causal_prefill_past_kv", choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time fa_bwd (dq, dk, dv) after one untimed forward; prefill workloads")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16"],
                    help="input type of q, k, v and out (fp16 peak = bf16 peak, as the nominal rates are equal)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
