"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The path shards by independent heads, so ranks exchange nothing on the data
path; what crosses ranks is the barrier around the timed region and the max
of the per-rank step times.  Each rank must draw a distinct batch.
"""
import os
import socket

import torch
import torch.multiprocessing as mp

import bench
from causal_linear_attention_attn_gb300 import inputs


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
