"""Shared helpers for GPU-vs-oracle parity tests.

Tolerance rule: max over the compared elements of |gpu - oracle| must not
exceed tau * RMS(oracle over the same elements), with tau = 1e-4 for float32
inputs and 2e-2 for bfloat16 inputs (fp32 accumulation, fp32 state).  The
same rule applies separately to out, S and z.
"""
import numpy as np
import torch

import oracle

TAU = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def err_ratio(gpu, ref) -> float:
    """max|gpu - ref| / RMS(ref)."""
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite GPU output (unwritten or overflowed element)"
    rms = np.sqrt(np.mean(r * r))
    return float(np.max(np.abs(g - r)) / rms) if r.size else 0.0


def assert_close(gpu, ref, tau, what=""):
    e = err_ratio(gpu, ref)
    assert e <= tau, f"{what}: max|err|/RMS = {e:.3g} > {tau:g}"
    return e


def oracle_seq(form, q, k, v, eps, nthreads=8, S0=None, z0=None):
    """Run the oracle on CPU copies of torch tensors [..., N, d]."""
    qd, kd, vd = f64(q), f64(k), f64(v)
    if form == "causal":
        return oracle.causal(qd, kd, vd, eps=eps, nthreads=nthreads, S0=S0, z0=z0)
    return oracle.global_(qd, kd, vd, eps=eps, nthreads=nthreads)
