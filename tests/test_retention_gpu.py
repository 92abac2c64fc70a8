"""GPU parity of retention (decayed state, no denominator) against the fp64 oracle.

Retention as "Linear Attention Math", "The kernel cousins: SSMs and RetNet"
states it: S_t = gamma_h S_{t-1} + k_t v_t^T and out_t = q_t^T S_t, q and k
used as given.  Two kernels serve it: the tensor-core causal pass in its
retention mode (bf16, d = 128, every decay at least 0.75) and an exact fp32
CUDA-core pass for everything else (fp32 inputs, d of 32 or 64, decays down
to 0).  Small cases compare every element of out and S, across shapes that
cut heads into segments both ways (first-pass CTAs aligned to the segments,
or flattened runs of two pieces), ragged tails, continuation from a given
state, the decays 0, 0.5, 0.75, 0.97 and 1, a prefill handed to the decode
step, and the full-size retention workload on sampled heads, all within the
float32 tolerance.
"""
import dataclasses

import numpy as np
import pytest
import torch

from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

import oracle

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS["retention_bf16"]
DEV = "cuda"
# The inputs are bf16, but every operand the kernel forms from them (the
# weighted scores, the weighted keys, the state copy read by the queries)
# reaches the tensor cores as a bf16 hi/lo pair (about 2^-17 relative) with
# fp32 accumulation, so the results meet the float32 inputs' bar.
TOL = TAU[torch.float32]


def _poison(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def _oracle(q, k, v, gamma, S0=None):
    B, H = q.shape[:2]
    g = np.tile(np.asarray(gamma, np.float64), B).reshape(B, H)
    return oracle.retention(f64(q), f64(k), f64(v), g, S0=S0, nthreads=8)


def _run(L, q, k, v, gamma):
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    out, S = _poison(B, H, N, dv), _poison(B, H, dk, dv)
    L.la_retention(q.to(DEV), k.to(DEV), v.to(DEV), gamma, out=out, S=S)
    torch.cuda.synchronize()
    return out, S


# (B, H, N): one chunk, ragged single segments, and heads split into segments
# whose first pass runs flattened (few heads) or aligned (38 heads of 1024 tokens)
SHAPES = [(1, 1, 1), (1, 2, 127), (1, 1, 128), (1, 3, 300), (2, 2, 1100), (1, 1, 2000), (3, 1, 4097),
          (2, 19, 1024), (1, 8, 5000)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_retention_every_element(cuda_lib, shape):
    B, H, N = shape
    q, k, v = inputs.make_qkv(W, N=N, B=B, H=H)
    gamma = inputs.retention_gamma(H)
    out, S = _run(cuda_lib, q, k, v, gamma)
    ro, rS = _oracle(q, k, v, gamma)
    assert_close(out, ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


@pytest.mark.parametrize("g", [0.75, 0.9, 1.0])
@pytest.mark.parametrize("N", [300, 2500])
def test_retention_fixed_decay(cuda_lib, g, N):
    q, k, v = inputs.make_qkv(W, N=N, B=1, H=2)
    out, S = _run(cuda_lib, q, k, v, [g, g])
    ro, rS = _oracle(q, k, v, [g, g])
    assert_close(out, ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


@pytest.mark.parametrize("split,N", [(1, 700), (128, 700), (200, 700), (1000, 3000), (129, 2200)])
def test_retention_with_state_continues_the_prefix(cuda_lib, split, N):
    q, k, v = inputs.make_qkv(W, N=N, B=1, H=3)
    gamma = inputs.retention_gamma(3)
    ro, rS = _oracle(q, k, v, gamma)
    d = lambda t: t.contiguous().to(DEV)
    L = cuda_lib
    o1, S = L.la_retention(d(q[:, :, :split]), d(k[:, :, :split]), d(v[:, :, :split]), gamma)
    o2, S = L.la_retention_with_state(d(q[:, :, split:]), d(k[:, :, split:]), d(v[:, :, split:]), S, gamma)
    torch.cuda.synchronize()
    assert_close(torch.cat([o1, o2], 2), ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_from_a_carried_state(cuda_lib):
    """Start from the oracle's state after an independent 1000-token prefix (a
    carried state of the same distribution), with decays from 0.75 to 1."""
    B, H, N = 1, 4, 1500
    q, k, v = inputs.make_qkv(W, N=N, B=B, H=H)
    gamma = [0.75, 0.95, 0.999, 1.0]
    _, kp, vp = inputs.make_qkv(dataclasses.replace(W, seed=W.seed + 1), N=1000, B=B, H=H)
    _, S0 = _oracle(kp, kp, vp, gamma)
    S0 = torch.from_numpy(S0).float()
    ro, rS = _oracle(q, k, v, gamma, S0=f64(S0))
    S = S0.to(DEV)
    out = _poison(B, H, N, 128)
    cuda_lib.la_retention_with_state(q.to(DEV), k.to(DEV), v.to(DEV), S, gamma, out=out)
    torch.cuda.synchronize()
    assert_close(out, ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_workload_full_size(cuda_lib):
    """The full retention workload on the GPU; every output of three sampled heads."""
    q, k, v = inputs.make_qkv(W)
    gamma = inputs.retention_gamma(W.H)
    out, S = _run(cuda_lib, q, k, v, gamma)
    heads = [0, 23, 63]
    qs, ks, vs = (t.view(W.BH, W.N, -1)[heads] for t in (q, k, v))
    g = [gamma[h % W.H] for h in heads]
    ro, rS = oracle.retention(f64(qs), f64(ks), f64(vs), np.asarray(g), nthreads=3)
    assert_close(out.view(W.BH, W.N, -1)[heads], ro, TOL, "out")
    assert_close(S.view(W.BH, 128, 128)[heads], rS, TOL, "S")
    assert torch.isfinite(out).all() and torch.isfinite(S).all()


def test_retention_edge_cases(cuda_lib):
    L = cuda_lib
    e = torch.empty(2, 3, 0, 128, dtype=torch.bfloat16, device=DEV)
    out, S = L.la_retention(e, e, e, [0.9] * 3, S=_poison(2, 3, 128, 128))
    torch.cuda.synchronize()
    assert out.shape == (2, 3, 0, 128) and torch.count_nonzero(S) == 0
    S0 = torch.randn(2, 3, 128, 128, device=DEV)
    S1 = S0.clone()
    L.la_retention_with_state(e, e, e, S1, [0.9] * 3)
    torch.cuda.synchronize()
    assert torch.equal(S0, S1)
    with pytest.raises(L.LinAttnError, match="UNSUPPORTED"):
        q = torch.zeros(1, 1, 8, 48, dtype=torch.bfloat16, device=DEV)
        L.la_retention(q, q, q, [0.9])
    with pytest.raises(L.LinAttnError, match="UNSUPPORTED"):
        q = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16, device=DEV)
        L.la_retention(q, q, q, [1.5])
    assert L.device_status() == 0


# --- the CUDA-core pass: fp32 inputs, d of 32 / 64, decays below 0.75 ----------

def _qkv(B, H, N, dk, dv, dtype, seed):
    """Retention-workload statistics at other sizes: q, k ~ N(0,1)/sqrt(d_k), v ~ N(0,1)."""
    gen = torch.Generator().manual_seed(seed)
    q, k = (torch.randn(B, H, N, dk, generator=gen) / dk ** 0.5 for _ in range(2))
    v = torch.randn(B, H, N, dv, generator=gen)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    return q.to(tdt), k.to(tdt), v.to(tdt)


CORE_GAMMA = [0.0, 0.5, 0.75, 0.97, 1.0]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (32, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("N", [1, 64, 200])
def test_retention_cuda_core_every_element(cuda_lib, dtype, dk, dv, N):
    """Decays 0 .. 1 across five heads, one chunk, an exact chunk and a ragged tail."""
    q, k, v = _qkv(2, 5, N, dk, dv, dtype, seed=N * 7 + dk + dv)
    out, S = _run(cuda_lib, q, k, v, CORE_GAMMA)
    ro, rS = _oracle(q, k, v, CORE_GAMMA)
    assert_close(out, ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_zero_decay_keeps_the_current_token(cuda_lib):
    """gamma = 0: out_t = (q_t . k_t) v_t and S = k_{N-1} v_{N-1}^T, from the definition alone."""
    q, k, v = _qkv(1, 1, 130, 64, 64, "f32", seed=5)
    out, S = _run(cuda_lib, q, k, v, [0.0])
    qd, kd, vd = (t[0, 0].double() for t in (q, k, v))
    want = (qd * kd).sum(-1, keepdim=True) * vd
    assert_close(out[0, 0], want.numpy(), TOL, "out")
    assert_close(S[0, 0], torch.outer(kd[-1], vd[-1]).numpy(), TOL, "S")


@pytest.mark.parametrize("N", [300, 2500])
def test_retention_decays_from_one_half_to_one(cuda_lib, N):
    """The retention workload's bf16 d = 128 inputs with decays 0.5, 0.75, 0.97 and 1."""
    gamma = [0.5, 0.75, 0.97, 1.0]
    q, k, v = inputs.make_qkv(W, N=N, B=1, H=4)
    out, S = _run(cuda_lib, q, k, v, gamma)
    ro, rS = _oracle(q, k, v, gamma)
    assert_close(out, ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


@pytest.mark.parametrize("split", [1, 64, 100])
def test_retention_cuda_core_with_state_continues_the_prefix(cuda_lib, split):
    gamma = [0.5, 0.9, 1.0]
    q, k, v = _qkv(2, 3, 300, 64, 32, "f32", seed=split)
    ro, rS = _oracle(q, k, v, gamma)
    d = lambda t: t.contiguous().to(DEV)
    L = cuda_lib
    o1, S = L.la_retention(d(q[:, :, :split]), d(k[:, :, :split]), d(v[:, :, :split]), gamma)
    o2, S = L.la_retention_with_state(d(q[:, :, split:]), d(k[:, :, split:]), d(v[:, :, split:]), S, gamma)
    torch.cuda.synchronize()
    assert_close(torch.cat([o1, o2], 2), ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_fast_decay_prefill_then_decode(cuda_lib):
    """A gamma = 0.5 prefill handed to the recurrent step equals the longer prefill."""
    B, H, N, steps = 2, 3, 700, 4
    gamma = [0.5, 0.5, 0.97]
    q, k, v = inputs.make_qkv(W, N=N + steps, B=B, H=H)
    ro, rS = _oracle(q, k, v, gamma)
    d = lambda t: t.contiguous().to(DEV)
    L = cuda_lib
    out, S = L.la_retention(d(q[:, :, :N]), d(k[:, :, :N]), d(v[:, :, :N]), gamma)
    outs = [out]
    for t in range(N, N + steps):
        outs.append(L.la_retention_decode_step(d(q[:, :, t]), d(k[:, :, t]), d(v[:, :, t]), S, gamma)[:, :, None])
    torch.cuda.synchronize()
    assert_close(torch.cat(outs, 2), ro, TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_cuda_core_full_size(cuda_lib):
    """The full retention workload with every other head at gamma = 0.5 (so the
    CUDA-core pass takes the whole call); every output of three sampled heads."""
    q, k, v = inputs.make_qkv(W)
    gamma = [0.5 if h % 2 else g for h, g in enumerate(inputs.retention_gamma(W.H))]
    out, S = _run(cuda_lib, q, k, v, gamma)
    heads = [0, 23, 63]
    qs, ks, vs = (t.view(W.BH, W.N, -1)[heads] for t in (q, k, v))
    g = [gamma[h % W.H] for h in heads]
    ro, rS = oracle.retention(f64(qs), f64(ks), f64(vs), np.asarray(g), nthreads=3)
    assert_close(out.view(W.BH, W.N, -1)[heads], ro, TOL, "out")
    assert_close(S.view(W.BH, 128, 128)[heads], rS, TOL, "S")


# --- the recurrent retention step ----------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (32, 128), (64, 64), (128, 32), (128, 128)])
def test_retention_decode_step_every_element(cuda_lib, dtype, dk, dv):
    """One step from a random state, decays 0 .. 1 across the heads; the step
    is fp32 arithmetic on the given inputs, so both dtypes meet the float32 bar."""
    B, H = 3, 5
    gen = torch.Generator().manual_seed(dk * 1000 + dv)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    q, k = (torch.randn(B, H, dk, generator=gen) / dk ** 0.5 for _ in range(2))
    v = torch.randn(B, H, dv, generator=gen)
    q, k, v = q.to(tdt), k.to(tdt), v.to(tdt)
    S0 = torch.randn(B, H, dk, dv, generator=gen)
    gamma = [0.0, 0.5, 0.9, 0.999, 1.0]
    ro, rS = _oracle(q[:, :, None], k[:, :, None], v[:, :, None], gamma, S0=f64(S0))
    S = S0.to(DEV)
    out = cuda_lib.la_retention_decode_step(q.to(DEV), k.to(DEV), v.to(DEV), S, gamma)
    torch.cuda.synchronize()
    assert_close(out, ro[:, :, 0], TOL, "out")
    assert_close(S, rS, TOL, "S")


def test_retention_prefill_then_decode_equals_longer_prefill(cuda_lib):
    B, H, N, steps = 2, 3, 700, 4
    q, k, v = inputs.make_qkv(W, N=N + steps, B=B, H=H)
    gamma = inputs.retention_gamma(H)
    ro, rS = _oracle(q, k, v, gamma)
    d = lambda t: t.contiguous().to(DEV)
    L = cuda_lib
    out, S = L.la_retention(d(q[:, :, :N]), d(k[:, :, :N]), d(v[:, :, :N]), gamma)
    outs = [out]
    for t in range(N, N + steps):
        outs.append(L.la_retention_decode_step(d(q[:, :, t]), d(k[:, :, t]), d(v[:, :, t]), S, gamma)[:, :, None])
    torch.cuda.synchronize()
    assert_close(torch.cat(outs, 2), ro, TOL, "out")
    assert_close(S, rS, TOL, "S")
