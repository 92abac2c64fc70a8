"""GPU parity: the C-ABI CUDA path against the fp64 oracle on the same seeded inputs.

Small cases compare every element; the five full-size workloads run on the
GPU at full size (the launch the benchmark times) and compare every output
of sampled heads, whose oracle runs token by token on the CPU.
"""
import dataclasses

import numpy as np
import pytest
import torch

from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64, oracle_seq

import oracle

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS
DEV = "cuda"


def _poison(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def _run(L, form, q, k, v, eps):
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    out, S, z = _poison(B, H, N, dv), _poison(B, H, dk, dv), _poison(B, H, dk)
    fn = L.la_causal if form == "causal" else L.la_global
    fn(q.to(DEV), k.to(DEV), v.to(DEV), out=out, S=S, z=z, eps=eps)
    torch.cuda.synchronize()
    return out, S, z


SMALL = [(1, 1, 1, 32, 32), (1, 2, 63, 64, 32), (2, 1, 129, 32, 128), (1, 3, 300, 128, 128),
         (1, 2, 1000, 128, 64), (2, 2, 257, 64, 64), (1, 1, 640, 128, 128),
         # d = 128 bf16 shapes that split heads into several segments, with ragged tails
         (1, 1, 2000, 128, 128), (1, 2, 1100, 128, 128), (3, 1, 4097, 128, 128), (1, 1, 127, 128, 128)]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("form", ["causal", "global"])
def test_small_shapes_every_element(cuda_lib, form, dtype, shape):
    B, H, N, dk, dv = shape
    base = W["causal_f32_small"] if dtype == "f32" else W["causal_bf16"]
    w = dataclasses.replace(base, dk=dk, dv=dv)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    out, S, z = _run(cuda_lib, form, q, k, v, w.eps)
    ro, rS, rz = oracle_seq(form, q, k, v, w.eps)
    tau = TAU[w.torch_dtype]
    assert_close(out, ro, tau, "out")
    assert_close(S, rS, tau, "S")
    assert_close(z, rz, tau, "z")


# Tensor-core global form (bf16, d_k = d_v in {64, 128}): clusters of 1 to 8 CTAs
# per head in the state build, persistent read CTAs that cross many heads.
GLOBAL_TC = [(1, 1, 1, 64), (1, 1, 8192, 64), (1, 1, 16384, 64), (2, 3, 129, 64), (4, 40, 200, 64),
             (10, 100, 100, 64), (1, 2, 5000, 128), (2, 2, 383, 128), (1, 1, 1, 128), (3, 60, 130, 128),
             # d = 64 with more heads than half the SMs and fewer than all (one build CTA a head),
             # ragged tails
             (1, 100, 1000, 64), (3, 40, 257, 64), (1, 151, 128, 64), (2, 50, 4161, 64), (1, 77, 64, 64),
             # d = 64 with a CTA per head covering at least 80 % of the SMs (the one-pass kernel):
             # more tiles than the read's stages and the build's slots, ragged tails, one token
             (2, 64, 1000, 64), (1, 130, 1537, 64), (1, 122, 3000, 64), (3, 50, 700, 64), (1, 128, 1, 64)]


@pytest.mark.parametrize("shape", GLOBAL_TC, ids=lambda s: "x".join(map(str, s)))
def test_global_tensor_core_shapes_every_element(cuda_lib, shape):
    B, H, N, d = shape
    w = dataclasses.replace(W["global_bf16"], dk=d, dv=d)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    out, S, z = _run(cuda_lib, "global", q, k, v, w.eps)
    ro, rS, rz = oracle_seq("global", q, k, v, w.eps)
    assert_close(out, ro, 2e-2, "out")
    assert_close(S, rS, 2e-2, "S")
    assert_close(z, rz, 2e-2, "z")
    assert cuda_lib.device_status() == 0


# Heads the planner cuts into two segments (51 to 76 heads on 152 SMs, at least 8 chunks):
# the second segment starts from the first pass's pieces.  Ragged tails, a one-token last
# chunk, and a carried state.
TWO_SEGMENT = [(1, 64, 1000, False), (2, 30, 3000, False), (1, 76, 2049, False), (1, 64, 1300, True)]


@pytest.mark.parametrize("shape", TWO_SEGMENT, ids=lambda s: "x".join(map(str, s)))
def test_two_segment_heads_every_element_of_sampled_heads(cuda_lib, shape):
    B, H, N, from_state = shape
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    g = torch.Generator().manual_seed(11)
    S0 = torch.randn(B, H, 128, 128, generator=g) if from_state else None
    z0 = torch.rand(B, H, 128, generator=g) * 50 + 1 if from_state else None
    if from_state:
        S, z = S0.to(DEV), z0.to(DEV)
        out, _, _ = cuda_lib.la_causal_with_state(q.to(DEV), k.to(DEV), v.to(DEV), S, z, eps=w.eps)
    else:
        out, S, z = cuda_lib.la_causal(q.to(DEV), k.to(DEV), v.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    heads = [0, 1, B * H - 2, B * H - 1]
    sel = lambda t: t.reshape(B * H, *t.shape[2:])[heads]
    ro, rS, rz = oracle.causal(f64(sel(q)), f64(sel(k)), f64(sel(v)), eps=w.eps, nthreads=4,
                               S0=f64(sel(S0)) if from_state else None, z0=f64(sel(z0)) if from_state else None)
    assert_close(sel(out), ro, 2e-2, "out")
    assert_close(sel(S), rS, 2e-2, "S")
    assert_close(sel(z), rz, 2e-2, "z")


def test_workload_causal_f32_small_every_element(cuda_lib):
    w = W["causal_f32_small"]
    q, k, v = inputs.make_qkv(w)
    out, S, z = _run(cuda_lib, "causal", q, k, v, w.eps)
    ro, rS, rz = oracle_seq("causal", q, k, v, w.eps)
    assert_close(out, ro, 1e-4, "out")
    assert_close(S, rS, 1e-4, "S")
    assert_close(z, rz, 1e-4, "z")


def _full_size_sampled(L, name, heads):
    w = W[name]
    q, k, v = inputs.make_qkv(w)
    out, S, z = _run(L, w.form, q, k, v, w.eps)
    qs, ks, vs = (t.view(w.BH, w.N, -1)[heads] for t in (q, k, v))
    ro, rS, rz = oracle_seq(w.form, qs, ks, vs, w.eps, nthreads=len(heads))
    tau = TAU[w.torch_dtype]
    e = assert_close(out.view(w.BH, w.N, -1)[heads], ro, tau, f"{name} out")
    assert_close(S.view(w.BH, w.dk, w.dv)[heads], rS, tau, f"{name} S")
    assert_close(z.view(w.BH, w.dk)[heads], rz, tau, f"{name} z")
    assert torch.isfinite(out).all(), "an output element was never written"
    return e


def test_workload_global_bf16_full_size(cuda_lib):
    _full_size_sampled(cuda_lib, "global_bf16", [0, 37, 90, 127])


def test_workload_causal_bf16_full_size(cuda_lib):
    _full_size_sampled(cuda_lib, "causal_bf16", [0, 21, 63])


@pytest.mark.slow
def test_workload_causal_bf16_long_full_size(cuda_lib):
    _full_size_sampled(cuda_lib, "causal_bf16_long", [0, 31])


def test_workload_decode_full_size(cuda_lib):
    """Full decode batch: state from the 1024-token prefix (la_causal), then steps."""
    w = W["decode_bf16"]
    L = cuda_lib
    kp, vp = inputs.decode_prefix(w)
    kd, vd = kp.to(DEV), vp.to(DEV)
    _, S, z = L.la_causal(kd, kd, vd, eps=w.eps)  # prefix queries do not touch the state
    del kd, vd
    rng = np.random.default_rng(5)
    heads = sorted(rng.choice(w.BH, size=64, replace=False).tolist())
    _, rS, rz = oracle.causal(f64(kp.view(w.BH, w.prefix, -1)[heads]), f64(kp.view(w.BH, w.prefix, -1)[heads]),
                              f64(vp.view(w.BH, w.prefix, -1)[heads]), eps=w.eps, nthreads=8)
    for step in range(6):
        q, k, v = inputs.decode_step_qkv(w, step)
        out = _poison(w.B, w.H, w.dv)
        L.la_decode_step(q.to(DEV), k.to(DEV), v.to(DEV), S, z, out=out, eps=w.eps)
        ro, rS, rz = oracle.decode_step(f64(q.view(w.BH, -1)[heads]), f64(k.view(w.BH, -1)[heads]),
                                        f64(v.view(w.BH, -1)[heads]), rS, rz, eps=w.eps)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert_close(out.view(w.BH, -1)[heads], ro, 2e-2, f"step {step} out")
    assert_close(S.view(w.BH, w.dk, w.dv)[heads], rS, 2e-2, "S")
    assert_close(z.view(w.BH, w.dk)[heads], rz, 2e-2, "z")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (32, 128), (64, 64), (64, 128), (128, 32), (128, 128)])
def test_decode_every_element_from_random_state(cuda_lib, dtype, dk, dv):
    base = W["causal_f32_small"] if dtype == "f32" else W["decode_bf16"]
    w = dataclasses.replace(base, dk=dk, dv=dv)
    B, H = 3, 5
    g = torch.Generator().manual_seed(11)
    S0 = torch.randn(B, H, dk, dv, generator=g) * 30
    z0 = torch.rand(B, H, dk, generator=g) * 1000 + 1
    S, z = S0.to(DEV), z0.to(DEV)
    rS, rz = f64(S0), f64(z0)
    for step in range(3):
        q, k, v = inputs.decode_step_qkv(w, step, B=B, H=H)
        out = cuda_lib.la_decode_step(q.to(DEV), k.to(DEV), v.to(DEV), S, z, eps=w.eps)
        ro, rS, rz = oracle.decode_step(f64(q), f64(k), f64(v), rS, rz, eps=w.eps)
        torch.cuda.synchronize()
        assert_close(out, ro, TAU[w.torch_dtype], "out")
    assert_close(S, rS, TAU[w.torch_dtype], "S")
    assert_close(z, rz, TAU[w.torch_dtype], "z")


# --- cross-form invariants on the GPU path ------------------------------------

def test_causal_last_row_and_state_equal_global(cuda_lib):
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=777, B=1, H=3)
    oc, Sc, zc = _run(cuda_lib, "causal", q, k, v, w.eps)
    og, Sg, zg = _run(cuda_lib, "global", q, k, v, w.eps)
    assert_close(oc[:, :, -1], f64(og[:, :, -1]), 2e-2, "last row")
    assert_close(Sc, f64(Sg), 2e-2, "S")
    assert_close(zc, f64(zg), 2e-2, "z")


def test_causal_prefix_then_decode_equals_longer_causal(cuda_lib):
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=300, B=2, H=2)
    ref, _, _ = oracle_seq("causal", q, k, v, w.eps)
    _, S, z = cuda_lib.la_causal(q[:, :, :290].contiguous().to(DEV), k[:, :, :290].contiguous().to(DEV),
                                 v[:, :, :290].contiguous().to(DEV), eps=w.eps)
    for t in range(290, 300):
        o = cuda_lib.la_decode_step(q[:, :, t].contiguous().to(DEV), k[:, :, t].contiguous().to(DEV),
                                    v[:, :, t].contiguous().to(DEV), S, z, eps=w.eps)
        torch.cuda.synchronize()
        assert_close(o, ref[:, :, t], 2e-2, f"token {t}")


@pytest.mark.parametrize("split,N", [(1, 700), (64, 700), (200, 700), (511, 700), (1000, 3000), (129, 2200)])
def test_causal_with_state_continues_the_prefix(cuda_lib, split, N):
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=N, B=1, H=2)
    ref, rS, rz = oracle_seq("causal", q, k, v, w.eps)
    d = lambda t: t.contiguous().to(DEV)
    o1, S, z = cuda_lib.la_causal(d(q[:, :, :split]), d(k[:, :, :split]), d(v[:, :, :split]), eps=w.eps)
    o2, S, z = cuda_lib.la_causal_with_state(d(q[:, :, split:]), d(k[:, :, split:]), d(v[:, :, split:]), S, z,
                                             eps=w.eps)
    torch.cuda.synchronize()
    assert_close(torch.cat([o1, o2], 2), ref, 2e-2, "out")
    assert_close(S, rS, 2e-2, "S")
    assert_close(z, rz, 2e-2, "z")


# --- edge cases ---------------------------------------------------------------

@pytest.mark.parametrize("form", ["causal", "global"])
def test_empty_sequence_writes_zero_state(cuda_lib, form):
    q = torch.zeros(2, 3, 0, 64, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(2, 3, 0, 32, dtype=torch.bfloat16, device=DEV)
    S, z = _poison(2, 3, 64, 32), _poison(2, 3, 64)
    fn = cuda_lib.la_causal if form == "causal" else cuda_lib.la_global
    out, S, z = fn(q, q, v, S=S, z=z)
    torch.cuda.synchronize()
    assert out.shape == (2, 3, 0, 32)
    assert torch.equal(S, torch.zeros_like(S)) and torch.equal(z, torch.zeros_like(z))


def test_empty_continuation_keeps_state(cuda_lib):
    q = torch.zeros(1, 2, 0, 32, dtype=torch.float32, device=DEV)
    S = torch.randn(1, 2, 32, 32, device=DEV)
    z = torch.rand(1, 2, 32, device=DEV)
    S0, z0 = S.clone(), z.clone()
    cuda_lib.la_causal_with_state(q, q, q, S, z)
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(z, z0)


def test_no_heads_is_a_no_op(cuda_lib):
    q = torch.zeros(0, 4, 16, 32, dtype=torch.bfloat16, device=DEV)
    out, S, z = cuda_lib.la_causal(q, q, q)
    assert out.numel() == 0


def test_large_magnitude_inputs_stay_finite(cuda_lib):
    """phi(x) = x + 1 grows linearly and exp(x) underflows to 0 for very negative x;
    the denominator stays positive as long as some feature is positive."""
    w = dataclasses.replace(W["causal_bf16"], qk_scale=8.0)
    q, k, v = inputs.make_qkv(w, N=200, B=1, H=2)
    out, S, z = _run(cuda_lib, "causal", q, k, v, w.eps)
    ro, rS, rz = oracle_seq("causal", q, k, v, w.eps)
    assert_close(out, ro, 2e-2, "out")


def test_no_bounded_wait_timed_out(cuda_lib):
    """Every tensor-core call above finished without a device-side wait giving up."""
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=1500, B=1, H=2)
    _run(cuda_lib, "causal", q, k, v, w.eps)
    assert cuda_lib.device_status() == 0
