"""fp64 CPU oracle for normalized (ELU+1) linear attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``la_oracle.c`` (plain C, double precision,
token-serial); this module only marshals numpy arrays.  Sources for every
formula are cited in that file's header:

* causal prefill (inclusive read): "线性注意力从头到尾讲清楚" §7; "Linear
  Attention: Accumulating KV in a Fixed-Size State", "Summarize state
  updates and reads with equations"; "Linear Attention Math", "The recurrent
  form".
* global read: "线性注意力从头到尾讲清楚" §5 and §8; "Linear Attention Math",
  "The associativity trick, written out".
* decode step: one update-then-read of the causal recurrence on a persistent
  state ("线性注意力从头到尾讲清楚" §7, last paragraph; "Linear Attention
  Math", "The recurrent form").
* retention: "Linear Attention Math", "The kernel cousins: SSMs and RetNet".
* positive random features: "Linear Attention Math", "Feature maps: elu+1
  and positive random features"; "线性注意力从头到尾讲清楚" §9.
* causal backward: the derivative of the causal definition (the pages name
  training through the chunked form but write no backward pass); pinned by
  finite differences of the forward.

Arrays: q, k are ``[..., N, dk]``; v is ``[..., N, dv]``; leading dimensions
are flattened into independent heads.  Results are float64.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, library_path

PHI_KINDS = {"elu1": 0, "identity": 1}

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(
            os.path.join(os.path.dirname(__file__), "la_oracle.c")
        ):
            build_oracle()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.lao_phi.argtypes = [D, I]
        lib.lao_phi.restype = D
        lib.lao_causal.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, L, L, I, I, D, I, I]
        lib.lao_causal.restype = I
        lib.lao_global.argtypes = [dp, dp, dp, dp, dp, dp, L, L, I, I, D, I, I]
        lib.lao_global.restype = I
        lib.lao_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, L, I, I, D, I, I]
        lib.lao_decode_step.restype = I
        lib.lao_state_scalars.argtypes = [I, I]
        lib.lao_retention.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, I, I, I]
        lib.lao_retention.restype = I
        lib.lao_causal_backward.argtypes = [dp] * 13 + [L, L, I, I, D, I, I]
        lib.lao_causal_backward.restype = I
        lib.lao_favor_features.argtypes = [dp, dp, dp, L, I, I]
        lib.lao_favor_features.restype = I
        lib.lao_state_scalars.restype = L
        lib.lao_version.restype = I
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name} failed with status {rc}")


def phi(x, kind: str = "elu1"):
    """Feature map applied elementwise (scalar or array)."""
    lib = _load()
    arr = np.asarray(x, dtype=np.float64)
    out = np.array([lib.lao_phi(float(t), PHI_KINDS[kind]) for t in arr.ravel()])
    return out.reshape(arr.shape) if arr.shape else float(out[0])


def _split(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim < 2 or q.shape != k.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("q, k must be [..., N, dk] and v [..., N, dv] with equal leading dims")
    lead = q.shape[:-2]
    N, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    return q, k, v, lead, BH, N, dk, dv


def causal(q, k, v, eps: float = 1e-6, phi: str = "elu1", S0=None, z0=None, nthreads: int = 1):
    """Causal prefill.  Returns (out [..., N, dv], S [..., dk, dv], z [..., dk])."""
    lib = _load()
    q, k, v, lead, BH, N, dk, dv = _split(q, k, v)
    out = np.empty(lead + (N, dv))
    S = np.empty(lead + (dk, dv))
    z = np.empty(lead + (dk,))
    S0 = None if S0 is None else _f64(np.broadcast_to(S0, lead + (dk, dv)))
    z0 = None if z0 is None else _f64(np.broadcast_to(z0, lead + (dk,)))
    rc = lib.lao_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z), _ptr(S0), _ptr(z0),
                        BH, N, dk, dv, float(eps), PHI_KINDS[phi], int(nthreads))
    _check(rc, "causal")
    return out, S, z


def global_(q, k, v, eps: float = 1e-6, phi: str = "elu1", nthreads: int = 1):
    """Global (non-causal) form.  Returns (out, S, z) like :func:`causal`."""
    lib = _load()
    q, k, v, lead, BH, N, dk, dv = _split(q, k, v)
    out = np.empty(lead + (N, dv))
    S = np.empty(lead + (dk, dv))
    z = np.empty(lead + (dk,))
    rc = lib.lao_global(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z),
                        BH, N, dk, dv, float(eps), PHI_KINDS[phi], int(nthreads))
    _check(rc, "global")
    return out, S, z


def decode_step(q, k, v, S, z, eps: float = 1e-6, phi: str = "elu1", nthreads: int = 1):
    """One decode step.  q, k: [..., dk]; v: [..., dv]; S: [..., dk, dv]; z: [..., dk].

    Returns (out [..., dv], S_new, z_new); the inputs S, z are not modified.
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-1]
    dk, dv = q.shape[-1], v.shape[-1]
    if k.shape != q.shape or v.shape[:-1] != lead:
        raise ValueError("decode_step: q, k must be [..., dk] and v [..., dv]")
    S = _f64(S).copy()
    z = _f64(z).copy()
    if S.shape != lead + (dk, dv) or z.shape != lead + (dk,):
        raise ValueError("decode_step: S must be [..., dk, dv] and z [..., dk]")
    BH = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (dv,))
    rc = lib.lao_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z),
                             BH, dk, dv, float(eps), PHI_KINDS[phi], int(nthreads))
    _check(rc, "decode_step")
    return out, S, z


def retention(q, k, v, gamma, S0=None, nthreads: int = 1):
    """Causal retention with decay: S_t = gamma S_{t-1} + k_t v_t^T, out_t = q_t^T S_t.

    q, k: [..., N, dk]; v: [..., N, dv]; gamma: a scalar, or one value per
    leading index (per head).  Returns (out [..., N, dv], S [..., dk, dv]).
    """
    lib = _load()
    q, k, v, lead, BH, N, dk, dv = _split(q, k, v)
    g = _f64(np.broadcast_to(np.asarray(gamma, dtype=np.float64), lead))
    out = np.empty(lead + (N, dv))
    S = np.empty(lead + (dk, dv))
    S0 = None if S0 is None else _f64(np.broadcast_to(S0, lead + (dk, dv)))
    rc = lib.lao_retention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(S0), _ptr(g), BH, N, dk, dv,
                           int(nthreads))
    _check(rc, "retention")
    return out, S


def state_scalars(m: int, dv: int) -> int:
    """Persistent state size per head (matrix plus normalizer vector)."""
    return int(_load().lao_state_scalars(m, dv))


def causal_backward(q, k, v, dout, eps: float = 1e-6, phi: str = "elu1", S0=None, z0=None, dS=None, dz=None,
                    nthreads: int = 1):
    """Gradients of the causal prefill for the upstream gradient ``dout`` of its
    output (and, optionally, ``dS``, ``dz`` of its final state).

    Returns (dq, dk, dv, dS0, dz0): the gradients w.r.t. q, k, v and the
    initial state (S0, z0; zero when the forward started from zero).
    """
    lib = _load()
    q, k, v, lead, BH, N, dk, dv = _split(q, k, v)
    dout = _f64(dout)
    if dout.shape != v.shape:
        raise ValueError("causal_backward: dout must have v's shape")
    bc = lambda a, shape: None if a is None else _f64(np.broadcast_to(a, shape))
    S0, dS = bc(S0, lead + (dk, dv)), bc(dS, lead + (dk, dv))
    z0, dz = bc(z0, lead + (dk,)), bc(dz, lead + (dk,))
    dq, dkk, dvv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
    dS0, dz0 = np.empty(lead + (dk, dv)), np.empty(lead + (dk,))
    rc = lib.lao_causal_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(S0), _ptr(z0), _ptr(dS), _ptr(dz),
                                 _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dS0), _ptr(dz0), BH, N, dk, dv, float(eps),
                                 PHI_KINDS[phi], int(nthreads))
    _check(rc, "causal_backward")
    return dq, dkk, dvv, dS0, dz0


def favor_features(x, W):
    """Positive random features phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m) of every
    row of ``x`` ([..., d]) for the projections ``W`` ([m, d]); returns [..., m]."""
    lib = _load()
    x, W = _f64(x), _f64(W)
    d = x.shape[-1]
    if W.ndim != 2 or W.shape[1] != d:
        raise ValueError("favor_features: W must be [m, d] with x's last dimension d")
    m = W.shape[0]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    out = np.empty(x.shape[:-1] + (m,))
    _check(lib.lao_favor_features(_ptr(x), _ptr(W), _ptr(out), rows, d, m), "favor_features")
    return out
