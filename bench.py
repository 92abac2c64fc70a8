"""Benchmark of the GB300 normalized linear attention library.

One JSON line on rank 0.  The headline ``value`` is causal prefill
throughput (B*H*N tokens/s) on the B=4, H=16, N=8192, d=128 bf16 workload;
one step is one ``la_causal`` call on device-resident inputs.  The other
forms on the hot path (global read, long-context causal prefill, prefill
continued from a carried state, retention with per-head decay, the
recurrent decode step) are timed in the same run and reported under
``forms`` with their own roofline fractions.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--gpus N`` without a launcher starts N ranks itself through
torch.distributed.run (one process per GPU); under a launcher, N must match
WORLD_SIZE.

``--impl reference`` times the fp64 CPU oracle (token-serial recurrence) on
the host cores instead, on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own seeded batch (weak scaling,
no collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from causal_linear_attention_attn_gb300 import inputs  # noqa: E402

METRIC = "causal prefill tokens/s (B·H·N/s) & decode HBM GB/s, % of roofline, 1×GB300"
HEADLINE = "causal_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129e6


# --- distributed plumbing (host logic, covered by the gloo tests) -------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def launch_plan(gpus: int, env, argv):
    """How `bench.py --gpus N` runs: None to run in this process, else the command
    that starts N ranks (one process per GPU, as the driver's torchrun does).
    Under a launcher WORLD_SIZE must equal --gpus."""
    if "WORLD_SIZE" in env:
        world = int(env["WORLD_SIZE"])
        if world != gpus:
            raise SystemExit(f"bench.py: --gpus {gpus} but the launcher started {world} ranks")
        return None
    if gpus <= 1:
        return None
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def rank_workload(w: inputs.Workload, rank: int) -> inputs.Workload:
    """Each rank draws its own batch (weak scaling): same shapes, distinct seed."""
    return dataclasses.replace(w, seed=w.seed + 7919 * rank) if rank else w


# --- roofline bookkeeping ------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def in_bytes(w):
    return 4 if w.dtype == "f32" else 2


def seq_bytes(w) -> float:
    """Algorithmic HBM bytes of one prefill/global call: q,k,v read, fp32 out
    written, final fp32 S and z written."""
    tok = w.BH * w.N
    return tok * (2 * w.dk + w.dv) * in_bytes(w) + tok * w.dv * 4 + w.BH * (w.dk * w.dv + w.dk) * 4


def decode_bytes(w) -> float:
    """Algorithmic HBM bytes of one decode step: S and z read and written (fp32),
    q,k,v read, fp32 out written."""
    return w.BH * (2 * (w.dk * w.dv + w.dk) * 4 + (2 * w.dk + w.dv) * in_bytes(w) + w.dv * 4)


def ncu_traffic(kernel_key: str):
    """Per-launch DRAM bytes measured by ncu for this kernel, if the kernel
    source is unchanged since the capture (see profiles/traffic.json)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    import hashlib

    h = hashlib.sha256()
    for f in d["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return d["bytes_per_launch"] if h.hexdigest()[:16] == d["sha"] else None


# --- clocks --------------------------------------------------------------------

class ClockSampler:
    """SM clock, power and throttle reasons sampled every few milliseconds while
    the bench runs (read-only queries).  NVML through ctypes when the driver's
    library loads, else `nvidia-smi --loop-ms` (100 ms period)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clocks-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.002

    def __init__(self, index: int):
        self.index, self.samples, self.proc, self.nvml, self.source = index, [], None, None, None
        self.stop = threading.Event()

    def _nvml_open(self):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        dev = ctypes.c_void_p()
        idx = self.index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        if ids and all(x.strip().isdigit() for x in ids) and self.index < len(ids):
            idx = int(ids[self.index])
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(dev)) != 0:
            raise OSError("no NVML handle")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.nvml = (ctypes, lib, dev, reasons)
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def _nvml_loop(self):
        ctypes, lib, dev, reasons = self.nvml
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            lib.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk))  # NVML_CLOCK_SM
            lib.nvmlDeviceGetPowerUsage(dev, ctypes.byref(mw))
            reasons(dev, ctypes.byref(rs))
            names = [n for bit, n in self.REASONS.items() if rs.value & bit]
            self.samples.append((time.time(), float(clk.value), mw.value / 1e3, names))
            time.sleep(self.PERIOD_S)

    def _smi_loop(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx, pw = float(f[0]), float(f[1]), float(f[2])
            except ValueError:
                continue
            self.max_mhz = mx
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            self.samples.append((time.time(), sm, pw, [n for n, v in zip(names, f[5:9]) if v.lower() == "active"]))

    def __enter__(self):
        self.max_mhz = None
        try:
            self._nvml_open()
            self.source = f"nvml every {self.PERIOD_S * 1e3:.0f} ms"
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
        except (OSError, AttributeError):
            self.nvml = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                return self
            self.source = "nvidia-smi every 100 ms"
            self.t = threading.Thread(target=self._smi_loop, daemon=True)
        self.t.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.source:
            self.t.join(timeout=2)
        if self.nvml:
            self.nvml[1].nvmlShutdown()

    def summary(self, t0: float, t1: float):
        """Clock record of the timed window [t0, t1].  A window shorter than the
        sampling period can hold no sample; then the samples within 20 ms of it
        are used (the GPU is busy with the same kernels just before and after)
        and the record says so."""
        rows = [r for r in self.samples if t0 <= r[0] <= t1]
        widened = not rows
        if widened:
            rows = [r for r in self.samples if t0 - 0.02 <= r[0] <= t1 + 0.02]
        if not rows:
            return None
        reasons = sorted({n for r in rows for n in r[3]})
        out = {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz,
               "power_w_max": round(max(r[2] for r in rows), 1), "samples": len(rows), "reasons": reasons,
               "source": self.source}
        if widened:
            out["window"] = "timed region +-20 ms (shorter than the sampling period)"
        return out


# --- timing helpers ---------------------------------------------------------------

LAST_WINDOW = [0.0, 0.0]  # host wall-clock bounds of the last timed region


def time_device(fn, steps: int, warmup: int, world: int, stream, L=None):
    """ms per step over `steps` timed steps.  With the library binding `L`, a
    second run of the same `steps` steps follows with the library's per-kernel
    event pairs on (read back by kernel_table).  The pairs sit between
    kernels and keep a kernel from starting beside its predecessor, so the
    step time comes from the first run only."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    LAST_WINDOW[0] = time.time()
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    LAST_WINDOW[1] = time.time()
    barrier(world)
    ms = a.elapsed_time(b) / steps  # ms per step (this rank)
    if L is not None:
        L.profile_enable(True)
        for _ in range(steps):
            fn()
        L.profile_enable(False)
        torch.cuda.synchronize()
    return ms


def kernel_table(L, steps):
    """Per-kernel launches and mean device time over the last timed region."""
    rows = {}
    for name in L.KERNELS:
        ms, n = L.profile_read(name)
        if n:
            rows[name] = {"launches": n, "ms_per_launch": ms / n}
    tot = sum(r["ms_per_launch"] * r["launches"] for r in rows.values())
    for r in rows.values():
        r["share"] = round(r["ms_per_launch"] * r["launches"] / tot, 4) if tot else None
    return rows


def kernel_bytes(w, kernel: str) -> float:
    """Algorithmic HBM bytes of one launch of `kernel` on workload `w`: the
    operands it must read and the results it must write, each once."""
    ib = in_bytes(w)
    state = 4 * (w.dk * w.dv + w.dk)
    if kernel == "causal_main":  # all q, k, v; outputs except each head's exact leading rows; final state
        ne = min(w.N, 64) if w.form == "causal" else 0  # given features: no exact leading rows
        return w.BH * (w.N * (2 * w.dk + w.dv) * ib + (w.N - ne) * 4 * w.dv + state)
    if kernel == "retention_main":  # all q, k, v; every output row; final S (no normalizer)
        return w.BH * (w.N * (2 * w.dk + w.dv) * ib + w.N * 4 * w.dv + 4 * w.dk * w.dv)
    if kernel == "global_state":
        return w.BH * (w.N * (w.dk + w.dv) * ib + state)
    if kernel == "global_read":
        return w.BH * (w.N * w.dk * ib + state + w.N * 4 * w.dv)
    if kernel == "global_fused":  # q, k, v in, out and the state written
        return w.BH * (w.N * (2 * w.dk + w.dv) * ib + w.N * 4 * w.dv + state)
    if kernel == "decode":
        return decode_bytes(w)
    if kernel == "backward":
        return backward_bytes(w)
    if kernel == "favor":  # one launch: the rows of q (or k) in, their 128 features out, the projections
        return w.BH * w.N * (w.dk + 128) * ib + 128 * w.dk * ib
    return seq_bytes(w)


def roofline(alg_bytes: float, ms: float, hbm: float, src: str, traffic, kernel=None):
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
         "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": src,
         "alg_bytes_per_launch": alg_bytes}
    if kernel:
        r = {"kernel": kernel, "ms_per_launch": round(ms, 5), **r}
    return r


def dominant_roofline(L, w, steps, hbm, src, key):
    """Roofline of the kernel with the largest device time in the timed region,
    timed live with its own event pairs, plus the per-kernel table."""
    table = kernel_table(L, steps)
    name = max(table, key=lambda n: table[n]["ms_per_launch"] * table[n]["launches"])
    t = table[name]
    return roofline(kernel_bytes(w, name), t["ms_per_launch"], hbm, src, ncu_traffic(f"{key}:{name}"),
                    kernel=name), table


# --- our arm -----------------------------------------------------------------------

def run_seq_form(L, w, steps, warmup, world, stream, hbm, src, gen_device="cuda"):
    q, k, v = inputs.make_qkv(w, device=gen_device)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(w.B, w.H, w.N, w.dv, dtype=torch.float32, device="cuda")
    S = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device="cuda")
    z = torch.empty(w.B, w.H, w.dk, dtype=torch.float32, device="cuda")
    # fn(q, k, v, out, S, z, h0): one call on heads [h0, h0 + q.shape[1]) of the flattened batch
    if w.form == "retention":
        gam = inputs.retention_gamma(w.H)
        fn = lambda q_, k_, v_, o_, S_, z_, h0: L.la_retention(
            q_, k_, v_, [gam[(h0 + i) % w.H] for i in range(q_.shape[1])], out=o_, S=S_, stream=stream)
    else:
        f = L.la_causal if w.form == "causal" else L.la_global
        fn = lambda q_, k_, v_, o_, S_, z_, h0: f(q_, k_, v_, out=o_, S=S_, z=z_, eps=w.eps, stream=stream)
    call = lambda: fn(q, k, v, out, S, z, 0)
    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (2 * steps + warmup) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    tok = w.BH * w.N
    rl, table = dominant_roofline(L, w, steps, hbm, src, w.name)
    step_bytes = retention_bytes(w) if w.form == "retention" else seq_bytes(w)
    res = {"workload": w.name, "tokens_per_s": world * tok / (ms * 1e-3), "ms_per_call": ms,
           "roofline": rl, "step_roofline": roofline(step_bytes, ms, hbm, src, None),
           "kernels": table, "gpu_launches": launches}
    return res, (q, k, v, out, S, z, fn)


def run_continue(L, w, steps, warmup, world, stream, hbm, src):
    """Prefill that continues from a carried state (la_causal_with_state): the
    state a call leaves is the state the next call starts from."""
    q, k, v = (t.cuda() for t in inputs.make_qkv(w, device="cuda"))
    out, S, z = L.la_causal(q, k, v, eps=w.eps, stream=stream)
    call = lambda: L.la_causal_with_state(q, k, v, S, z, out=out, eps=w.eps, stream=stream)
    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (2 * steps + warmup) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    rl, table = dominant_roofline(L, w, steps, hbm, src, w.name + "_with_state")
    step_bytes = seq_bytes(w) + w.BH * (w.dk * w.dv + w.dk) * 4  # the incoming state is read too
    return {"workload": w.name + " continued from a carried state", "tokens_per_s": world * w.BH * w.N / (ms * 1e-3),
            "ms_per_call": ms, "roofline": rl, "step_roofline": roofline(step_bytes, ms, hbm, src, None),
            "kernels": table, "gpu_launches": launches}


def run_e2e(L, w, bufs, steps, warmup, stream, groups: int = 4):
    """Same call through host buffers: every step copies q, k, v in from pinned
    host memory and out, S, z back.  The heads go through in `groups` groups
    on three streams (copy in, compute, copy out), so that the copies of one
    group overlap the call on another; a step still ends only when all of its
    results are on the host."""
    q, k, v, out, S, z, fn = bufs
    BH = w.BH
    flat = lambda t: t.view(BH, *t.shape[2:])
    dev = [flat(t) for t in (q, k, v, out, S, z)]
    host = [t.cpu().pin_memory() for t in dev[:3]] + [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                                                      for t in dev[3:]]
    cuts = [BH * g // groups for g in range(groups + 1)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        done_in = [torch.cuda.Event() for _ in range(groups)]
        done_call = [torch.cuda.Event() for _ in range(groups)]
        for g in range(groups):
            a, b = cuts[g], cuts[g + 1]
            with torch.cuda.stream(s_in):
                for d, h in zip(dev[:3], host[:3]):
                    d[a:b].copy_(h[a:b], non_blocking=True)
                done_in[g].record(s_in)
        for g in range(groups):
            a, b = cuts[g], cuts[g + 1]
            stream.wait_event(done_in[g])
            fn(*(t[a:b].unsqueeze(0) for t in dev), a)
            done_call[g].record(stream)
        for g in range(groups):
            a, b = cuts[g], cuts[g + 1]
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_call[g])
                for d, h in zip(dev[3:], host[3:]):
                    h[a:b].copy_(d[a:b], non_blocking=True)
        finished = torch.cuda.Event()
        finished.record(s_out)
        stream.wait_event(finished)

    ms = time_device(step, steps, warmup, 1, stream)
    h2d = sum(t.numel() * t.element_size() for t in host[:3])
    d2h = sum(t.numel() * t.element_size() for t in host[3:])
    return {"value": w.BH * w.N / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "head_groups": groups}


def run_decode(L, w, steps, warmup, world, stream, hbm, src):
    kp, vp = inputs.decode_prefix(w, device="cuda")
    S, z = L.la_causal(kp, kp, vp, eps=w.eps, stream=stream)[1:]
    del kp, vp
    torch.cuda.empty_cache()  # only the state stays on the device
    nstage = steps + warmup
    staged = [inputs.decode_step_qkv(w, s, device="cuda") for s in range(nstage)]
    out = torch.empty(w.B, w.H, w.dv, dtype=torch.float32, device="cuda")
    it = itertools.cycle(staged)  # the per-kernel timing run after the timed steps reuses them
    call = lambda: L.la_decode_step(*next(it), S, z, out=out, eps=w.eps, stream=stream)
    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (nstage + steps) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    rl, table = dominant_roofline(L, w, steps, hbm, src, w.name)
    step = roofline(decode_bytes(w), ms, hbm, src, None)
    return {"workload": w.name, "us_per_step": ms * 1e3, "gbs": step["achieved"], "frac_hbm": step["frac"],
            "seq_tokens_per_s": world * w.B / (ms * 1e-3), "steps_timed": steps, "roofline": rl,
            "step_roofline": step, "kernels": table, "gpu_launches": launches}


def run_favor(L, w, steps, warmup, world, stream, hbm, src):
    """FAVOR+ causal prefill: positive random features of q and k (m = 128), then
    the normalized causal read on them."""
    q, k, v = (t.cuda() for t in inputs.make_qkv(w, device="cuda"))
    P = inputs.favor_projections(w, device="cuda")
    fq, fk = (torch.empty(w.B, w.H, w.N, 128, dtype=q.dtype, device="cuda") for _ in range(2))
    out = torch.empty(w.B, w.H, w.N, w.dv, dtype=torch.float32, device="cuda")
    S = torch.empty(w.B, w.H, 128, w.dv, dtype=torch.float32, device="cuda")
    z = torch.empty(w.B, w.H, 128, dtype=torch.float32, device="cuda")

    def call():
        L.la_favor_features(q, P, out=fq, stream=stream)
        L.la_favor_features(k, P, out=fk, stream=stream)
        L.la_causal_features(fq, fk, v, out=out, S=S, z=z, eps=w.eps, stream=stream)

    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (2 * steps + warmup) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    rl, table = dominant_roofline(L, w, steps, hbm, src, w.name)
    step_bytes = 2 * kernel_bytes(w, "favor") + seq_bytes(w)
    return {"workload": w.name, "tokens_per_s": world * w.BH * w.N / (ms * 1e-3), "ms_per_call": ms,
            "roofline": rl, "step_roofline": roofline(step_bytes, ms, hbm, src, None), "kernels": table,
            "gpu_launches": launches}


def backward_bytes(w) -> float:
    """Algorithmic HBM bytes of one causal backward: q, k, v and the fp32 upstream
    gradient read, fp32 dq, dk, dv written."""
    return w.BH * w.N * ((2 * w.dk + w.dv) * in_bytes(w) + 4 * w.dv + 4 * (2 * w.dk + w.dv))


# fp32 CUDA-core peak of a GB300: 152 SMs x 128 fp32 lanes x 2 FLOP per multiply-add x 2.07 GHz
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def backward_flops(w, chunk: int = 64) -> float:
    """FLOPs (2 per multiply-add) that a chunked causal backward needs: per token, five
    d_k x d_v state products (the fold S += phi(k) v^T; the read dO S^T, which serves
    both gden and dq; the fold U += phi(q) gnum^T; the state terms U v and U^T phi(k)
    of dk and dv), the intra-chunk scores phi(q).phi(k) and dO.v over one chunk,
    and the three products with a triangular operand at half a chunk."""
    per_token = 5 * w.dk * w.dv + chunk * (w.dk + w.dv) + chunk // 2 * (2 * w.dk + w.dv)
    return 2.0 * w.BH * w.N * per_token


def alu_roofline(flops: float, ms: float) -> dict:
    achieved = flops / (ms * 1e-3) / 1e12
    return {"bound": "alu", "achieved": round(achieved, 2), "peak": round(FP32_PEAK_TFLOPS, 1), "unit": "TFLOP/s",
            "frac": round(achieved / FP32_PEAK_TFLOPS, 4),
            "peak_source": "152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz", "alg_flops_per_call": flops}


def tensor_roofline(flops: float, ms: float) -> dict:
    """Algorithmic FLOPs per call against the measured dense bf16 tensor peak."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak, srcp = 1900.0, "fallback 1.9 PFLOP/s"
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        if m.get("bf16_tflops"):
            peak, srcp = float(m["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    achieved = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_source": srcp, "alg_flops_per_call": flops}


def run_backward(L, w, steps, warmup, world, stream, hbm, src):
    """Gradient of the causal prefill (la_causal_backward) for a seeded upstream gradient."""
    q, k, v = (t.cuda() for t in inputs.make_qkv(w, device="cuda"))
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 17)
    dO = torch.randn(w.B, w.H, w.N, w.dv, generator=g, device="cuda")
    call = lambda: L.la_causal_backward(q, k, v, dO, eps=w.eps, stream=stream)
    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (2 * steps + warmup) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    rl, table = dominant_roofline(L, w, steps, hbm, src, w.name + "_backward")
    tc = w.dtype == "bf16" and w.dk == w.dv == 128
    res = {"workload": w.name + " backward", "roofline": rl, "tokens_per_s": world * w.BH * w.N / (ms * 1e-3),
           "ms_per_call": ms, "step_roofline": roofline(backward_bytes(w), ms, hbm, src, None), "kernels": table,
           "gpu_launches": launches}
    if tc:
        res["tensor_roofline"] = tensor_roofline(backward_flops(w, chunk=128), ms)
        res["note"] = ("tcgen05 kernels, 128-token chunks, bf16 hi/lo operand pairs (about 3x the algorithmic "
                       "tensor work issued); pass 1 in order, pass 2 in reverse with dv and dk roles")
    else:
        res["alu_roofline"] = alu_roofline(backward_flops(w), ms)
        res["note"] = "exact fp32 CUDA-core kernel, each head cut into segments"
    return res


def retention_decode_bytes(w) -> float:
    """Algorithmic HBM bytes of one retention step: S read and written (fp32, no z),
    q,k,v read, fp32 out written."""
    return w.BH * (2 * w.dk * w.dv * 4 + (2 * w.dk + w.dv) * in_bytes(w) + w.dv * 4)


def run_retention_decode(L, w, steps, warmup, world, stream, hbm, src):
    """Retention step on the decode workload's batch: the state from a retention
    prefill over the same prefix, then one token per head per step."""
    kp, vp = inputs.decode_prefix(w, device="cuda")
    gamma = inputs.retention_gamma(w.H)
    S = L.la_retention(kp, kp, vp, gamma, stream=stream)[1]
    del kp, vp
    torch.cuda.empty_cache()  # only the state stays on the device
    nstage = steps + warmup
    staged = [inputs.decode_step_qkv(w, s, device="cuda") for s in range(nstage)]
    out = torch.empty(w.B, w.H, w.dv, dtype=torch.float32, device="cuda")
    it = itertools.cycle(staged)
    call = lambda: L.la_retention_decode_step(*next(it), S, gamma, out=out, stream=stream)
    n0 = L.kernel_launches()
    ms = time_device(call, steps, warmup, world, stream, L)
    launches = (L.kernel_launches() - n0) // (nstage + steps) * steps
    ms = max_over_ranks(ms, world, "cuda" if world > 1 else None)
    table = kernel_table(L, steps)
    t = table["retention_decode"]
    rl = roofline(retention_decode_bytes(w), t["ms_per_launch"], hbm, src, ncu_traffic(f"{w.name}:retention_decode"),
                  kernel="retention_decode")
    step = roofline(retention_decode_bytes(w), ms, hbm, src, None)
    return {"workload": "retention step on " + w.name, "us_per_step": ms * 1e3, "gbs": step["achieved"],
            "frac_hbm": step["frac"], "steps_timed": steps, "roofline": rl, "step_roofline": step, "kernels": table,
            "gpu_launches": launches}


def cpu_baseline(w, target_s: float = 12.0):
    """The oracle as it stands, token-serial fp64, heads spread over the host cores."""
    import numpy as np

    import oracle

    def run(q, k, v, nthreads):
        # heads 0 .. n-1 of the workload, as the oracle's form for it
        if w.form == "retention":
            g = inputs.retention_gamma(w.H)
            return oracle.retention(q, k, v, np.array([g[h % w.H] for h in range(q.shape[0])]), nthreads=nthreads)
        fn = oracle.causal if w.form == "causal" else oracle.global_
        return fn(q, k, v, eps=w.eps, nthreads=nthreads)

    cores = len(os.sched_getaffinity(0))
    # calibrate on a short prefix of one head, then size the sample
    q, k, v = inputs.make_qkv(w, N=min(w.N, 1024), heads=[0])
    t = time.perf_counter()
    run(q.double().numpy(), k.double().numpy(), v.double().numpy(), 1)
    per_tok = (time.perf_counter() - t) / q.shape[1]
    heads = max(1, min(w.BH, int(target_s * cores / (per_tok * w.N))))
    N = w.N if heads > 1 or per_tok * w.N * 1.0 <= target_s else max(1, int(target_s / per_tok))
    q, k, v = inputs.make_qkv(w, N=N, heads=list(range(min(heads, w.BH))))
    args = [np.ascontiguousarray(t.double().numpy()) for t in (q, k, v)]
    nthreads = min(cores, q.shape[0])
    t = time.perf_counter()
    run(*args, nthreads)
    dt = time.perf_counter() - t
    tok = q.shape[0] * q.shape[1]
    return {"value": tok / dt, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{q.shape[0]} of {w.BH} heads x {q.shape[1]} tokens of {w.name}, {dt:.1f} s wall"}


def retention_bytes(w) -> float:
    """Algorithmic HBM bytes of one retention call: q,k,v read, fp32 out and S written."""
    return w.BH * (w.N * (2 * w.dk + w.dv) * in_bytes(w) + w.N * 4 * w.dv + 4 * w.dk * w.dv)


def decode_workload(args):
    """The decode workload, with its batch reduced by --decode-batch (small profiling runs)."""
    w = inputs.WORKLOADS["decode_bf16"]
    return dataclasses.replace(w, B=args.decode_batch) if args.decode_batch else w


# Forms on the bench line, in this order: a reader of only the line's end (a log that keeps its
# tail) sees the long-context causal form, the global form and the decode step last.
FORM_ORDER = ("causal_bf16_backward", "favor_bf16", "retention_bf16", "causal_bf16_with_state",
              "retention_decode_bf16", "decode_bf16", "global_bf16", "causal_bf16_long")


def compact(res: dict) -> dict:
    """The figures of one form that the bench line carries: step time, rate, step
    roofline fraction, and the dominant kernel's name, live time, fraction and
    traffic (launch counts and clocks are in the --detail record; clock throttle
    reasons, if any, are kept here)."""
    rl, step = res["roofline"], res["step_roofline"]
    c = {"ms": round(res.get("ms_per_call", res.get("us_per_step", 0.0) / 1e3), 5)}
    if "tokens_per_s" in res:
        c["tokens_per_s"] = float(f"{res['tokens_per_s']:.4g}")
    if "gbs" in res:
        c["gbs"] = res["gbs"]
    c["step_frac"] = step["frac"]
    c["kernel"] = rl["kernel"]
    c["kernel_ms"] = rl["ms_per_launch"]
    c["kernel_frac"] = rl["frac"]
    if rl.get("traffic"):
        c["traffic"] = rl["traffic"]
    if "alu_roofline" in res:
        c["alu_frac"] = res["alu_roofline"]["frac"]
    if "tensor_roofline" in res:
        c["tensor_frac"] = res["tensor_roofline"]["frac"]
    clk = res.get("clocks") or {}
    if clk.get("reasons"):
        c["clock_reasons"] = clk["reasons"]
    return c


def ordered_forms(forms: dict) -> dict:
    names = [n for n in FORM_ORDER if n in forms] + [n for n in forms if n not in FORM_ORDER]
    return {n: compact(forms[n]) for n in names}


def carry_study(args):
    """Times the causal prefill with each head carried by one CTA (G = 1) and cut
    into G segments (the first pass's pieces start each segment), G as forced by
    la_diag_force_segments, against the planner's choice (G = 0), on the causal
    workloads.  Prints one JSON line with the step times."""
    torch.cuda.set_device(0)
    from causal_linear_attention_attn_gb300 import linattn as L

    hbm, src = peaks()
    stream = torch.cuda.current_stream()
    rows = {}
    for name in ("causal_bf16", "causal_bf16_long"):
        w = inputs.WORKLOADS[name]
        for G in (0, 1, 2, 4, 8, 16):
            if name == "causal_bf16_long" and G in (2, 4):
                continue
            L.diag_force_segments(G)
            try:
                r, _ = run_seq_form(L, w, max(3, args.steps // (10 if name == "causal_bf16_long" else 1)),
                                    args.warmup, 1, stream, hbm, src)
            finally:
                L.diag_force_segments(0)
            rows[f"{name} G={G or 'auto'}"] = {"ms": round(r["ms_per_call"], 4),
                                               "step_frac": r["step_roofline"]["frac"],
                                               "kernels": {k: round(v["ms_per_launch"], 4)
                                                           for k, v in r["kernels"].items()}}
            torch.cuda.empty_cache()
    print(json.dumps({"carry_study": rows}))


def dry_run(args):
    """The multi-rank plumbing without a GPU (gloo): barrier, per-rank work, max over
    ranks and the whole-job value, printed by rank 0 in the bench line's shape."""
    world, rank, _ = dist_env()
    init_dist(world, "gloo")
    barrier(world)
    t = time.perf_counter()
    time.sleep(0.05 * (rank + 1))  # rank r "steps" for 50 (r + 1) ms
    ms = max_over_ranks((time.perf_counter() - t) * 1e3, world)
    barrier(world)
    if rank == 0:
        units = 1000  # per rank (weak scaling)
        print(json.dumps({"metric": METRIC, "dry_run": True, "n_gpus": world, "ms_per_step": ms,
                          "value": world * units / (ms * 1e-3), "scaling": "weak"}))
    if world > 1:
        torch.distributed.destroy_process_group()


def main_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    from causal_linear_attention_attn_gb300 import linattn as L

    hbm, src = peaks()
    stream = torch.cuda.current_stream()
    w = rank_workload(inputs.WORKLOADS[args.workload], rank)
    with ClockSampler(local) as clk:
        head, bufs = run_seq_form(L, w, args.steps, args.warmup, world, stream, hbm, src)
        t0, t1 = LAST_WINDOW
        forms = {}
        extras = [] if args.no_extras else [f for f in args.forms.split(",") if f]
        if not args.no_extras:
            for name in ("causal_bf16_long", "global_bf16"):
                if name == args.workload or name not in extras:
                    continue
                wx = rank_workload(inputs.WORKLOADS[name], rank)
                steps = max(3, args.steps // (10 if name == "causal_bf16_long" else 1))
                forms[name], _ = run_seq_form(L, wx, steps, args.warmup, world, stream, hbm, src)
                forms[name]["clocks"] = clk.summary(*LAST_WINDOW)
                torch.cuda.empty_cache()
        if "causal_bf16_with_state" in extras:
            wc = rank_workload(inputs.WORKLOADS["causal_bf16"], rank)
            forms["causal_bf16_with_state"] = run_continue(L, wc, max(3, args.steps // 2), args.warmup, world, stream,
                                                           hbm, src)
            forms["causal_bf16_with_state"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
        if "retention_bf16" in extras and args.workload != "retention_bf16":
            wr = rank_workload(inputs.WORKLOADS["retention_bf16"], rank)
            forms["retention_bf16"], _ = run_seq_form(L, wr, args.steps, args.warmup, world, stream, hbm, src)
            forms["retention_bf16"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
        if "favor_bf16" in extras:
            wf = rank_workload(inputs.WORKLOADS["favor_bf16"], rank)
            forms["favor_bf16"] = run_favor(L, wf, args.steps, args.warmup, world, stream, hbm, src)
            forms["favor_bf16"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
        if "causal_bf16_backward" in extras:
            wb = rank_workload(inputs.WORKLOADS["causal_bf16"], rank)
            forms["causal_bf16_backward"] = run_backward(L, wb, 3, args.warmup, world, stream, hbm, src)
            forms["causal_bf16_backward"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
        if "decode_bf16" in extras:
            wd = rank_workload(decode_workload(args), rank)
            forms["decode_bf16"] = run_decode(L, wd, args.decode_steps, args.warmup, world, stream, hbm, src)
            forms["decode_bf16"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
        if "retention_decode_bf16" in extras:
            wd = rank_workload(decode_workload(args), rank)
            forms["retention_decode_bf16"] = run_retention_decode(L, wd, args.decode_steps, args.warmup, world,
                                                                  stream, hbm, src)
            forms["retention_decode_bf16"]["clocks"] = clk.summary(*LAST_WINDOW)
            torch.cuda.empty_cache()
    e2e = run_e2e(L, w, bufs, max(3, args.steps // 10), args.warmup, stream, args.e2e_groups)
    cpu = cpu_baseline(w) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if rank != 0:
        return
    clocks = clk.summary(t0, t1)
    ms = head["ms_per_call"]
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded torch.randn, per-head seeds; drawn on the device)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_k": w.dk, "d_v": w.dv, "eps": w.eps,
                   "inputs": "q,k ~ N(0,1)/sqrt(128), v ~ N(0,1), bf16; out/S/z fp32",
                   "l2": "inputs (402.7 MB) larger than L2 (129 MB); no flush needed",
                   "parallelism": f"replicas x{world} (heads independent)"},
        "roofline": head["roofline"], "step_roofline": head["step_roofline"],
        "gpu_launches": head["gpu_launches"], "e2e": e2e, "clocks": clocks,
        "cpu_baseline": cpu,
        # every other form, compact and last on the line (long-context causal and global at the very end)
        "forms": ordered_forms(forms),
    }
    if args.detail:
        with open(args.detail, "w") as f:
            json.dump(dict(line, kernels=head["kernels"], forms=forms), f, indent=1)
    print(json.dumps(line))


# --- reference arm: the oracle on the host cores -------------------------------------

def main_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    # each step is a bounded sample sized so that the whole run stays near two minutes
    step_s = max(0.2, min(args.ref_step_s, 120.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, target_s=step_s)
    vals = [cpu_baseline(w, target_s=step_s) for _ in range(args.steps)]
    v = statistics.median(r["value"] for r in vals)
    cb = dict(vals[0], value=v)
    line = {"metric": METRIC, "impl": "reference", "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch.randn)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_k": w.dk, "d_v": w.dv},
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--decode-batch", type=int, default=0, help="decode forms: batch instead of 256 (profiling)")
    ap.add_argument("--no-extras", action="store_true", help="time the headline workload only")
    ap.add_argument("--forms", default="global_bf16,causal_bf16_long,causal_bf16_with_state,retention_bf16,favor_bf16,"
                                     "causal_bf16_backward,decode_bf16,retention_decode_bf16",
                    help="comma-separated other forms timed after the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=4, help="head groups the end-to-end leg pipelines over")
    ap.add_argument("--ref-step-s", type=float, default=10.0, help="max CPU seconds per reference step")
    ap.add_argument("--detail", default="", help="also write every form's full record (kernel tables) to this file")
    ap.add_argument("--dry-run", action="store_true", help="multi-rank plumbing only, on CPU (gloo); no GPU work")
    ap.add_argument("--carry-study", action="store_true",
                    help="time the causal prefill at forced segment counts (one JSON line; not the bench line)")
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    return a


if __name__ == "__main__":
    a = parse()
    cmd = launch_plan(a.gpus, os.environ, sys.argv[1:])
    if cmd is not None:  # --gpus N without a launcher: start N ranks like the driver's torchrun
        sys.exit(subprocess.call(cmd))
    if a.dry_run:
        dry_run(a)
    elif a.carry_study:
        carry_study(a)
    elif a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
