"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The path shards by independent heads, so ranks exchange nothing on the data
path; what crosses ranks is the barrier around the timed region and the max
of the per-rank step times.  Each rank must draw a distinct batch.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
from causal_linear_attention_attn_gb300 import inputs
from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w_, r_, l_ = bench.dist_env()
    assert (w_, r_, l_) == (world, rank, rank)
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 + rank, world)
    w = bench.rank_workload(inputs.WORKLOADS["causal_bf16"], rank)
    qv, _, _ = inputs.make_qkv(w, N=4, heads=[0])
    q.put((rank, m, w.seed, qv.float().sum().item()))
    torch.distributed.destroy_process_group()


def test_two_ranks_max_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == 2.5  # both ranks see the slowest rank's time
    assert res[0][2] != res[1][2]  # distinct seeds per rank
    assert res[0][3] != res[1][3]  # hence distinct data


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.rank_workload(inputs.WORKLOADS["causal_bf16"], 0) == inputs.WORKLOADS["causal_bf16"]


def test_algorithmic_bytes_of_the_workloads():
    W = inputs.WORKLOADS
    assert abs(bench.seq_bytes(W["causal_bf16"]) / 1e6 - 675.3) < 0.1
    assert abs(bench.seq_bytes(W["causal_bf16_long"]) / 1e6 - 5370.8) < 0.1
    assert abs(bench.seq_bytes(W["global_bf16"]) / 1e6 - 337.7) < 0.1
    assert abs(bench.decode_bytes(W["decode_bf16"]) / 1e6 - 1092.6) < 0.1


def test_backward_arithmetic_roofline():
    # d = 128, 64-token chunks: 5 d^2 + 64 (2 d) + 32 (3 d) = 110,592 multiply-adds per token
    w = inputs.WORKLOADS["causal_bf16"]
    assert bench.backward_flops(w) == 2.0 * 4 * 16 * 8192 * 110592
    assert abs(bench.FP32_PEAK_TFLOPS - 80.55) < 0.01
    r = bench.alu_roofline(bench.backward_flops(w), 5.0)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 2.0 * 4 * 16 * 8192 * 110592 / 5e-3 / 1e12) < 0.01
    assert abs(r["frac"] - r["achieved"] / bench.FP32_PEAK_TFLOPS) < 1e-3


def test_launch_plan_of_gpus_flag():
    """--gpus N without a launcher starts N ranks (torch.distributed.run, one per GPU);
    under a launcher the rank count must match."""
    cmd = bench.launch_plan(2, {}, ["--gpus", "2", "--steps", "3"])
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and "--master-addr=127.0.0.1" in cmd
    assert cmd[-4:] == [os.path.abspath(bench.__file__), "--gpus", "2", "--steps", "3"][-4:]
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}, []) is None
    assert bench.launch_plan(1, {}, []) is None
    with pytest.raises(SystemExit):
        bench.launch_plan(4, {"WORLD_SIZE": "2"}, [])


def test_gpus_two_runs_two_ranks_and_takes_the_slowest():
    """`bench.py --gpus 2 --dry-run` on CPU: two gloo ranks, rank 1 the slower (100 ms
    against 50 ms); rank 0 prints one line with n_gpus 2 and the whole-job value over
    the max time."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["dry_run"]
    assert line["ms_per_step"] >= 100.0
    assert abs(line["value"] - 2 * 1000 / (line["ms_per_step"] * 1e-3)) < 1e-6 * line["value"]
