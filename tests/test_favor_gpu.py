"""GPU parity of positive random features (la_favor_features) and of the
causal read on given features (la_causal_features) against the fp64 oracle.

The features are phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m) ("Linear
Attention Math", "Feature maps: elu+1 and positive random features").  The
feature map is checked element by element: the kernel's only rounding is
the bf16 (or fp32) output, so every feature must be within 2^-8 (bf16) or
1e-5 (fp32) of the oracle's, relative.  The causal read on given features is
checked against the oracle's identity-map causal form on the same features
(1e-4 of the RMS for fp32 inputs, 2e-2 for bf16).  The two together (FAVOR+ causal attention, features
stored in bf16 as the tensor-core read takes them) are checked on the
workload's shape with sampled heads against the oracle's features rounded
to bf16 and its read in fp64.  (Against unrounded fp64 features the
deviation is set by that storage: at the workload's scale the weights
concentrate on a few keys, so one feature's 2^-9 rounding moves an output
directly, to about 2e-2 of the RMS.)
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
W = inputs.WORKLOADS["favor_bf16"]


def _rel_err(got, ref):
    g = f64(got)
    assert np.all(np.isfinite(g))
    return float(np.max(np.abs(g - ref) / np.abs(ref)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d,m", [(128, 128), (64, 128), (128, 64), (32, 32), (128, 256), (64, 256)])
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_features_every_element(cuda_lib, dtype, d, m, N):
    w = dataclasses.replace(W, dk=d, dv=d, dtype=dtype)
    q, _, _ = inputs.make_qkv(w, N=N, B=1, H=3)
    P = inputs.favor_projections(w, m=m)
    phi = cuda_lib.la_favor_features(q.to(DEV), P.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.favor_features(f64(q), f64(P))
    assert phi.shape == (1, 3, N, m)
    assert _rel_err(phi, ref) <= (2.0 ** -8 if dtype == "bf16" else 1e-5)


# (B, H, N, m, d_v); m = 256 is the m = 2d setting (32-token chunks on the CUDA cores)
SHAPES = [(1, 1, 1, 128, 128), (1, 2, 300, 128, 128), (1, 1, 2000, 128, 128), (3, 1, 4097, 128, 128),
          (2, 19, 1024, 128, 128), (1, 2, 700, 64, 128), (2, 1, 129, 32, 64), (1, 2, 300, 256, 128),
          (2, 1, 65, 256, 32), (1, 1, 1, 256, 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_causal_on_given_features_every_element(cuda_lib, shape, dtype):
    """The read on the GPU's own features against the identity-map oracle on them."""
    B, H, N, m, dv = shape
    w = dataclasses.replace(W, dk=128, dv=dv, dtype=dtype)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    P = inputs.favor_projections(w, m=m).to(DEV)
    fq, fk = cuda_lib.la_favor_features(q.to(DEV), P), cuda_lib.la_favor_features(k.to(DEV), P)
    out, S, z = cuda_lib.la_causal_features(fq, fk, v.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    ro, rS, rz = oracle.causal(f64(fq), f64(fk), f64(v), eps=w.eps, phi="identity", nthreads=8)
    tau = TAU[w.torch_dtype]
    assert_close(out, ro, tau, "out")
    assert_close(S, rS, tau, "S")
    assert_close(z, rz, tau, "z")


@pytest.mark.parametrize("shape", [(1, 2, 300, 128, 128), (2, 3, 1000, 64, 128), (1, 1, 129, 32, 32),
                                   (1, 2, 300, 256, 128), (2, 1, 63, 256, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_global_on_given_features_every_element(cuda_lib, shape, dtype):
    B, H, N, m, dv = shape
    w = dataclasses.replace(W, dk=128, dv=dv, dtype=dtype)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    P = inputs.favor_projections(w, m=m).to(DEV)
    fq, fk = cuda_lib.la_favor_features(q.to(DEV), P), cuda_lib.la_favor_features(k.to(DEV), P)
    out, S, z = cuda_lib.la_global_features(fq, fk, v.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    ro, rS, rz = oracle.global_(f64(fq), f64(fk), f64(v), eps=w.eps, phi="identity", nthreads=8)
    tau = TAU[w.torch_dtype]
    assert_close(out, ro, tau, "out")
    assert_close(S, rS, tau, "S")
    assert_close(z, rz, tau, "z")


def test_favor_causal_end_to_end_workload_shape(cuda_lib):
    """The workload (4 x 16 x 8192, d = m = 128, bf16): features and read on the
    GPU; every output of three sampled heads against the oracle's features of
    the same inputs, stored in bf16 as the GPU stores them, and its fp64 read."""
    q, k, v = inputs.make_qkv(W)
    P = inputs.favor_projections(W)
    Pd = P.to(DEV)
    fq, fk = cuda_lib.la_favor_features(q.to(DEV), Pd), cuda_lib.la_favor_features(k.to(DEV), Pd)
    out, S, z = cuda_lib.la_causal_features(fq, fk, v.to(DEV), eps=W.eps)
    torch.cuda.synchronize()
    heads = [0, 33, 63]
    sel = lambda t: f64(t.reshape(W.BH, W.N, -1)[heads])
    bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    rq, rk = bf16(oracle.favor_features(sel(q), f64(P))), bf16(oracle.favor_features(sel(k), f64(P)))
    ro, rS, rz = oracle.causal(rq, rk, sel(v), eps=W.eps, phi="identity", nthreads=3)
    assert_close(out.reshape(W.BH, W.N, -1)[heads], ro, TAU[torch.bfloat16], "out")
    assert_close(S.reshape(W.BH, 128, 128)[heads], rS, TAU[torch.bfloat16], "S")
    assert torch.isfinite(out).all()
    assert cuda_lib.device_status() == 0


def test_favor_twice_the_features_end_to_end(cuda_lib):
    """m = 2d = 256 features of d = 128 bf16 inputs (two tensor-core feature launches), then the
    causal read on them (CUDA cores); every output against the oracle's bf16-stored features and
    its fp64 read, and every feature against the oracle's to 2^-8."""
    w = dataclasses.replace(W, B=1, H=4, N=1500)
    q, k, v = inputs.make_qkv(w)
    P = inputs.favor_projections(w, m=256)
    Pd = P.to(DEV)
    fq, fk = cuda_lib.la_favor_features(q.to(DEV), Pd), cuda_lib.la_favor_features(k.to(DEV), Pd)
    out, S, z = cuda_lib.la_causal_features(fq, fk, v.to(DEV), eps=w.eps)
    torch.cuda.synchronize()
    assert fq.shape == (1, 4, 1500, 256) and S.shape == (1, 4, 256, 128)
    rq64, rk64 = oracle.favor_features(f64(q), f64(P)), oracle.favor_features(f64(k), f64(P))
    assert _rel_err(fq, rq64) <= 2.0 ** -8 and _rel_err(fk, rk64) <= 2.0 ** -8
    bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    ro, rS, rz = oracle.causal(bf16(rq64), bf16(rk64), f64(v), eps=w.eps, phi="identity", nthreads=4)
    assert_close(out, ro, TAU[torch.bfloat16], "out")
    assert_close(S, rS, TAU[torch.bfloat16], "S")
    assert_close(z, rz, TAU[torch.bfloat16], "z")
    assert cuda_lib.device_status() == 0
