"""Seeded synthetic inputs for the seven workloads (no attention arithmetic here).

Every tensor is drawn as float32 ``torch.randn`` from a seeded generator,
multiplied by its scale, then rounded to the workload's input dtype
(bfloat16 rounds to nearest even).  Generation is per head: head ``bh`` of a
workload uses its own generator seeded with ``seed * 1_000_003 + bh`` and
draws q, k, v in that order, so any subset of heads can be regenerated on
its own for a spot check.  Decode steps draw one generator per step for all
heads.

``device="cuda"`` draws with torch's CUDA generator instead (same seeds,
different stream of numbers); the benchmark uses it to stage large inputs
quickly.  Parity tests always draw on the CPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    form: str  # "causal", "global", "retention", "favor" or "decode"
    B: int
    H: int
    N: int
    dk: int
    dv: int
    dtype: str  # "f32" or "bf16": dtype of q, k, v; outputs and state are float32
    qk_scale: float
    v_scale: float
    eps: float
    seed: int
    prefix: int = 0  # decode: tokens whose causal state initialises S, z
    prefix_scale: float = 1.0  # decode: scale of the prefix k, v draws
    steps: int = 0  # decode: consecutive timed steps
    note: str = field(default="", compare=False)

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    w.name: w
    for w in [
        Workload("causal_f32_small", "causal", 1, 2, 256, 32, 32, "f32", 1.0, 1.0, 1e-6, 1001,
                 note="causal fp32, B=1 H=2 N=256 d=32, q,k,v ~ N(0,1)"),
        Workload("global_bf16", "global", 8, 16, 4096, 64, 64, "bf16", 1 / math.sqrt(64), 1.0, 1e-6, 1002,
                 note="global bf16, B=8 H=16 N=4096 d=64, q,k ~ N(0,1)/sqrt(64), v ~ N(0,1)"),
        Workload("causal_bf16", "causal", 4, 16, 8192, 128, 128, "bf16", 1 / math.sqrt(128), 1.0, 1e-6, 1003,
                 note="causal prefill bf16, B=4 H=16 N=8192 d=128, q,k ~ N(0,1)/sqrt(128), v ~ N(0,1)"),
        Workload("causal_bf16_long", "causal", 1, 32, 131072, 128, 128, "bf16", 1 / math.sqrt(128), 1.0, 1e-6,
                 1004, note="long-context causal prefill bf16, B=1 H=32 N=131072 d=128"),
        Workload("retention_bf16", "retention", 4, 16, 8192, 128, 128, "bf16", 1 / math.sqrt(128), 1.0, 0.0, 1006,
                 note="retention bf16, B=4 H=16 N=8192 d=128, q,k ~ N(0,1)/sqrt(128), v ~ N(0,1), "
                      "gamma_h = 1 - 2^-(5 + h mod 8)"),
        Workload("favor_bf16", "favor", 4, 16, 8192, 128, 128, "bf16", 128 ** -0.25, 1.0, 1e-6, 1007,
                 note="causal prefill on positive random features, B=4 H=16 N=8192 d=128, m=128 projections "
                      "W ~ N(0,1); q,k ~ N(0,1)/128^(1/4) (the softmax kernel exp(q.k/sqrt(d))), v ~ N(0,1)"),
        Workload("decode_bf16", "decode", 256, 32, 1, 128, 128, "bf16", 1 / math.sqrt(128), 1.0, 1e-6, 1005,
                 prefix=1024, prefix_scale=1.0, steps=1000,
                 note="decode step, batch 256 H=32 m=d_v=128, fp32 state from a 1024-token N(0,1) prefix"),
    ]
}


def retention_gamma(H: int) -> list[float]:
    """Per-head decays of the retention inputs: gamma_h = 1 - 2^-(5 + h mod 8).

    Eight scales from 0.96875 (a key's weight halves in about 22 tokens) to
    1 - 2^-12 (about 2800 tokens), repeated over the heads; every value is
    exact in float32.
    """
    return [1.0 - 2.0 ** -(5 + h % 8) for h in range(H)]


def favor_projections(w: Workload, m: int = 128, device: str = "cpu"):
    """The m random projections of the positive random features, [m, d] ~ N(0, 1),
    drawn from the workload's seed and rounded to its input dtype."""
    return _draw((m, w.dk), 1.0, w.torch_dtype, _gen(w.seed * 1_000_003 + 70_000_000, device), device)


def _gen(seed: int, device: str):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _draw(shape, scale, dtype, g, device):
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def head_qkv(w: Workload, bh: int, N: int | None = None, scale_qk=None, scale_v=None,
             dtype=None, device: str = "cpu", seed_offset: int = 0):
    """q [N, dk], k [N, dk], v [N, dv] of head ``bh`` (flattened b*H + h)."""
    N = w.N if N is None else N
    dtype = w.torch_dtype if dtype is None else dtype
    sq = w.qk_scale if scale_qk is None else scale_qk
    sv = w.v_scale if scale_v is None else scale_v
    g = _gen(w.seed * 1_000_003 + bh + seed_offset, device)
    q = _draw((N, w.dk), sq, dtype, g, device)
    k = _draw((N, w.dk), sq, dtype, g, device)
    v = _draw((N, w.dv), sv, dtype, g, device)
    return q, k, v


def make_qkv(w: Workload, N: int | None = None, heads=None, device: str = "cpu", B: int | None = None,
             H: int | None = None):
    """Whole-batch q, k, v shaped [B, H, N, d] in the workload's input dtype.

    ``heads`` restricts generation to a list of flattened head indices
    (returned stacked as [len(heads), N, d]).  ``B``/``H`` override the
    batch shape (same per-head seeds), for reduced-size cases.
    """
    N = w.N if N is None else N
    B = w.B if B is None else B
    H = w.H if H is None else H
    idx = list(range(B * H)) if heads is None else list(heads)
    qs, ks, vs = [], [], []
    for bh in idx:
        q, k, v = head_qkv(w, bh, N, device=device)
        qs.append(q), ks.append(k), vs.append(v)
    q, k, v = torch.stack(qs), torch.stack(ks), torch.stack(vs)
    if heads is None:
        q = q.view(B, H, N, w.dk)
        k = k.view(B, H, N, w.dk)
        v = v.view(B, H, N, w.dv)
    return q, k, v


def decode_prefix(w: Workload, heads=None, device: str = "cpu", B: int | None = None, H: int | None = None):
    """Prefix keys/values [.., prefix, d] whose causal state initialises the decode state.

    Drawn N(0,1) * prefix_scale in the workload dtype.  The prefix queries do
    not affect the state and are not drawn.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    idx = list(range(B * H)) if heads is None else list(heads)
    ks, vs = [], []
    for bh in idx:
        g = _gen(w.seed * 1_000_003 + 50_000_000 + bh, device)
        ks.append(_draw((w.prefix, w.dk), w.prefix_scale, w.torch_dtype, g, device))
        vs.append(_draw((w.prefix, w.dv), w.prefix_scale, w.torch_dtype, g, device))
    k, v = torch.stack(ks), torch.stack(vs)
    if heads is None:
        k = k.view(B, H, w.prefix, w.dk)
        v = v.view(B, H, w.prefix, w.dv)
    return k, v


def decode_step_qkv(w: Workload, step: int, device: str = "cpu", B: int | None = None, H: int | None = None):
    """Per-step q, k [B, H, dk] and v [B, H, dv] for decode step ``step``."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    g = _gen(w.seed * 1_000_003 + 90_000_000 + step, device)
    q = _draw((B, H, w.dk), w.qk_scale, w.torch_dtype, g, device)
    k = _draw((B, H, w.dk), w.qk_scale, w.torch_dtype, g, device)
    v = _draw((B, H, w.dv), w.v_scale, w.torch_dtype, g, device)
    return q, k, v
