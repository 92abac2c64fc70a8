"""GPU parity of the causal backward (la_causal_backward) against the fp64 oracle.

The oracle's gradient is the derivative of the causal definition, pinned by
finite differences of the forward (tests/test_oracle_backward_pins.py).

Two kernels compute it.  bf16 inputs with d_k = d_v = 128 take the tensor-core
kernel, whose products take bf16 operand pairs (about 16 significant bits)
with fp32 accumulation; it is held to the bar for bf16 inputs, max|err| <=
2e-2 RMS.  Every other case (fp32 inputs, other head sizes) takes the fp32
CUDA-core kernel, held to the float32 bar 1e-4 on sequences of up to 1000
tokens.  Cases: ragged shapes over every head size, a carried initial state
and a final-state gradient, the chain of two calls (the second call's
initial-state gradient fed to the first as its final-state gradient equals
the gradient of one long call), chunk-boundary lengths on the tensor-core
path, the headline workload's shape on sampled heads, and the empty and
degenerate cases.
"""
import dataclasses

import numpy as np
import pytest
import torch

from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = TAU[torch.float32]


def tol(dtype: str, dk: int, dv: int) -> float:
    """The bar of the kernel that takes the case: bf16 pairs on the tensor cores for
    bf16 inputs at d_k = d_v = 128, exact fp32 otherwise."""
    return TAU[torch.bfloat16] if dtype == "bf16" and dk == dv == 128 else TOL


def _grad_in(shape, seed):
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed))


def _state(B, H, dk, dv, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, dk, dv, generator=g), torch.rand(B, H, dk, generator=g) * 4 + 1


# heads cut into 1 to 8 segments (the backward spreads each head over about 152 / heads CTAs)
SHAPES = [(1, 1, 2, 32, 32), (1, 2, 63, 64, 32), (2, 1, 129, 32, 128), (1, 3, 300, 128, 128),
          (1, 2, 700, 128, 64), (2, 2, 257, 64, 64), (1, 1, 2000, 64, 64), (1, 2, 1500, 128, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_state", [False, True])
def test_backward_every_element(cuda_lib, shape, dtype, with_state):
    B, H, N, dk, dv = shape
    base = inputs.WORKLOADS["causal_f32_small" if dtype == "f32" else "causal_bf16"]
    w = dataclasses.replace(base, dk=dk, dv=dv)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    dO = _grad_in((B, H, N, dv), 100 + N)
    S0 = z0 = dS = dz = None
    if with_state:
        S0, z0 = _state(B, H, dk, dv, 7)
        dS, dz = _state(B, H, dk, dv, 8)
    d = lambda t: None if t is None else t.to(DEV)
    dq, dkk, dvv, dS0, dz0 = cuda_lib.la_causal_backward(d(q), d(k), d(v), d(dO), S0=d(S0), z0=d(z0), dS=d(dS),
                                                         dz=d(dz), need_state_grad=True, eps=w.eps)
    torch.cuda.synchronize()
    f = lambda t: None if t is None else f64(t)
    r = oracle.causal_backward(f64(q), f64(k), f64(v), f64(dO), eps=w.eps, S0=f(S0), z0=f(z0), dS=f(dS), dz=f(dz),
                               nthreads=8)
    for name, got, ref in zip(("dq", "dk", "dv", "dS0", "dz0"), (dq, dkk, dvv, dS0, dz0), r):
        assert_close(got, ref, tol(dtype, dk, dv), name)


# the tensor-core path at chunk boundaries (128 tokens) and across many chunks
TC_SHAPES = [(2, 1, 127), (1, 2, 128), (1, 1, 129), (1, 3, 255), (1, 1, 256), (2, 2, 1000), (1, 1, 3001)]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("with_state", [False, True])
def test_backward_tensor_core_lengths(cuda_lib, shape, with_state):
    B, H, N = shape
    w = inputs.WORKLOADS["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    dO = _grad_in((B, H, N, 128), 300 + N)
    S0 = z0 = dS = dz = None
    if with_state:
        S0, z0 = _state(B, H, 128, 128, 17)
        dS, dz = _state(B, H, 128, 128, 18)
    d = lambda t: None if t is None else t.to(DEV)
    outs = cuda_lib.la_causal_backward(d(q), d(k), d(v), d(dO), S0=d(S0), z0=d(z0), dS=d(dS), dz=d(dz),
                                       need_state_grad=True, eps=w.eps)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    f = lambda t: None if t is None else f64(t)
    r = oracle.causal_backward(f64(q), f64(k), f64(v), f64(dO), eps=w.eps, S0=f(S0), z0=f(z0), dS=f(dS), dz=f(dz),
                               nthreads=4)
    for name, got, ref in zip(("dq", "dk", "dv", "dS0", "dz0"), outs, r):
        assert_close(got, ref, TAU[torch.bfloat16], name)


@pytest.mark.parametrize("dtype,dv", [("f32", 64), ("bf16", 64), ("bf16", 128)])
def test_backward_single_token(cuda_lib, dtype, dv):
    """One token: o_0 = v_0 up to eps, so dv_0 = dO_0 (times 1 - eps/den) and the
    exact dq, dk are of order eps; on the GPU they are fp32 cancellation residue
    of S gnum against z gden, bounded here relative to dO (bf16 at d_v = 128 is
    the tensor-core path)."""
    base = inputs.WORKLOADS["causal_f32_small" if dtype == "f32" else "causal_bf16"]
    w = dataclasses.replace(base, dk=128, dv=dv)
    q, k, v = inputs.make_qkv(w, N=1, B=2, H=3)
    dO = _grad_in((2, 3, 1, dv), 5)
    dq, dkk, dvv = cuda_lib.la_causal_backward(q.to(DEV), k.to(DEV), v.to(DEV), dO.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    r = oracle.causal_backward(f64(q), f64(k), f64(v), f64(dO), eps=w.eps)
    assert_close(dvv, r[2], tol(dtype, 128, dv), "dv")
    scale = float(dO.pow(2).mean().sqrt())
    assert dq.abs().max().item() <= 1e-5 * scale and dkk.abs().max().item() <= 1e-5 * scale


def test_backward_chains_through_the_state(cuda_lib):
    """Backward of [prefix | rest]: the rest's initial-state gradient, passed to the
    prefix as its final-state gradient, gives the gradient of one long call."""
    w = inputs.WORKLOADS["causal_bf16"]
    B, H, N, split = 1, 2, 900, 333
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    dO = _grad_in((B, H, N, 128), 9)
    d = lambda t: t.contiguous().to(DEV)
    L = cuda_lib
    # the prefix's state from the oracle (exact), so that only the chaining is under test
    _, S1, z1 = oracle.causal(f64(q[:, :, :split]), f64(k[:, :, :split]), f64(v[:, :, :split]), eps=w.eps)
    S1, z1 = (torch.from_numpy(x).float().to(DEV) for x in (S1, z1))
    dq2, dk2, dv2, dS1, dz1 = L.la_causal_backward(d(q[:, :, split:]), d(k[:, :, split:]), d(v[:, :, split:]),
                                                   d(dO[:, :, split:]), S0=S1, z0=z1, need_state_grad=True, eps=w.eps)
    dq1, dk1, dv1 = L.la_causal_backward(d(q[:, :, :split]), d(k[:, :, :split]), d(v[:, :, :split]),
                                         d(dO[:, :, :split]), dS=dS1, dz=dz1, eps=w.eps)
    torch.cuda.synchronize()
    r = oracle.causal_backward(f64(q), f64(k), f64(v), f64(dO), eps=w.eps, nthreads=2)
    for name, a, b, ref in (("dq", dq1, dq2, r[0]), ("dk", dk1, dk2, r[1]), ("dv", dv1, dv2, r[2])):
        assert_close(torch.cat([a, b], 2), ref, tol("bf16", 128, 128), name)


def test_backward_headline_shape_sampled_heads(cuda_lib):
    """The causal headline's shape (4 x 16 x 8192, d = 128, bf16) on the GPU;
    every gradient of three sampled heads against the oracle."""
    w = inputs.WORKLOADS["causal_bf16"]
    q, k, v = inputs.make_qkv(w)
    dO = torch.randn(w.B, w.H, w.N, w.dv, generator=torch.Generator().manual_seed(11))
    dq, dkk, dvv = cuda_lib.la_causal_backward(q.to(DEV), k.to(DEV), v.to(DEV), dO.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    heads = [0, 29, 63]
    sel = lambda t: t.reshape(w.BH, w.N, -1)[heads]
    r = oracle.causal_backward(f64(sel(q)), f64(sel(k)), f64(sel(v)), f64(sel(dO)), eps=w.eps, nthreads=3)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dkk, dvv), r):
        assert_close(sel(got), ref, TAU[torch.bfloat16], name)
    assert torch.isfinite(dq).all() and torch.isfinite(dkk).all() and torch.isfinite(dvv).all()


def test_backward_edge_cases(cuda_lib):
    L = cuda_lib
    e = torch.empty(2, 3, 0, 64, device=DEV)
    dS, dz = torch.randn(2, 3, 64, 64, device=DEV), torch.randn(2, 3, 64, device=DEV)
    dq, dkk, dvv, dS0, dz0 = L.la_causal_backward(e, e, e, e, dS=dS, dz=dz, need_state_grad=True)
    torch.cuda.synchronize()
    assert dq.shape == (2, 3, 0, 64) and torch.equal(dS0, dS) and torch.equal(dz0, dz)
    # a zero upstream gradient gives zero gradients
    w = inputs.WORKLOADS["causal_f32_small"]
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(w, N=100, B=1, H=2))
    z = torch.zeros(1, 2, 100, 32, device=DEV)
    for g in L.la_causal_backward(q, k, v, z):
        assert torch.count_nonzero(g) == 0
    assert L.device_status() == 0


def test_backward_rows_not_32_byte_aligned(cuda_lib):
    """The tensor-core kernel moves rows 32 bytes at a time; inputs that are only
    16-byte aligned (what the ABI asks for) take the CUDA-core kernel instead and
    still match the oracle."""
    w = inputs.WORKLOADS["causal_bf16"]
    B, H, N = 1, 2, 300
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    dO = _grad_in((B, H, N, 128), 21)

    def shifted(t):  # the same values at an address 16 bytes past a 32-byte boundary
        n = t.numel()
        pad = 16 // t.element_size()
        buf = torch.empty(n + pad, dtype=t.dtype, device=DEV)
        out = buf[pad:].view(t.shape)
        out.copy_(t.to(DEV))
        assert out.data_ptr() % 32 == 16
        return out

    dq, dkk, dvv = cuda_lib.la_causal_backward(shifted(q), shifted(k), v.to(DEV), dO.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    r = oracle.causal_backward(f64(q), f64(k), f64(v), f64(dO), eps=w.eps, nthreads=2)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dkk, dvv), r):
        assert_close(got, ref, TAU[torch.bfloat16], name)
