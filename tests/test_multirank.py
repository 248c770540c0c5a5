"""Multi-rank host logic of the benchmark, as two gloo processes on the CPU.

Attention over independent sequences shards by replica: each rank runs the
whole path on its own batch (same shapes, its own seed), with no exchange on
the data path.  The only collectives are the timing ones: a barrier around the
timed region and a max over the ranks' times.  These tests run that logic with
world size 2 on gloo, and the reference arm under torch.distributed.run, where
rank 0 alone works and prints one line."""
import json
import os
import socket
import subprocess
import sys
import types

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench._dist()
    try:
        assert dist.get_backend() == "gloo"
        assert dist.get_rank() == rank and dist.get_world_size() == world
        # slowest rank decides the time, on every rank
        t = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
        # replicas: same shapes, different draws
        args = types.SimpleNamespace(workload="sliding_window_decode", seed=3, dtype="bf16")
        case = bench.replica_case(args, rank)
        shape = list(case["q"].shape) + list(case["k"].shape)
        digest = float(case["q"].float().sum() + 2 * case["k"].float().sum())
        got = [None] * world
        dist.all_gather_object(got, (shape, digest))
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max_ms": t, "gathered": got}, f)
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_timing_and_replicas(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [r["max_ms"] for r in res] == [15.0, 15.0]
    (s0, d0), (s1, d1) = res[0]["gathered"]
    assert s0 == s1
    assert d0 != d1


def test_job_value_counts_every_rank():
    import bench
    one = bench.job_value(2.0, 1, 4.0)
    assert one == 2.0 / 4e-3
    assert bench.job_value(2.0, 2, 4.0) == 2 * one
    assert bench.max_over_ranks(None, 7.5) == 7.5


def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "sliding_window_decode", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_line_keys():
    """The reference arm's line (one process): the contract's keys, the
    oracle as its own CPU baseline, and an e2e with no copies."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "sliding_window_decode",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["warmup"] >= 3
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert "workload" in line["config"]
