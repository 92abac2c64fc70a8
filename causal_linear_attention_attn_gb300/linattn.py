"""Thin ctypes binding of ``liblinattn.so`` (argument marshalling only).

Function names match the C ABI in ``include/linattn.h``.  Tensors are torch
CUDA tensors; the binding checks shapes and dtypes, allocates outputs that
were not supplied, passes raw device pointers and the current CUDA stream,
and raises :class:`LinAttnError` on a non-OK status.  Every step of the
computation runs in the library's kernels.  Importing this module fails if
the library has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblinattn.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() before use")

lib = ctypes.CDLL(LIB_PATH)

LA_F32, LA_BF16 = 0, 1
STATUS_NAMES = {0: "LA_OK", 1: "LA_ERR_INVALID_VALUE", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_MISALIGNED",
                4: "LA_ERR_OUT_OF_MEMORY", 5: "LA_ERR_LAUNCH", 6: "LA_ERR_TIMEOUT", 7: "LA_ERR_NO_DEVICE",
                8: "LA_ERR_TOO_LARGE"}

_vp, _fp, _i, _f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_SEQ_ARGS = [_vp, _vp, _vp, _fp, _fp, _fp, _i, _i, _i, _i, _i, _f, _i, _vp]
for _name in ("la_global", "la_causal", "la_causal_with_state", "la_causal_noalloc", "la_causal_features",
              "la_global_features"):
    getattr(lib, _name).argtypes = _SEQ_ARGS
    getattr(lib, _name).restype = _i
for _name in ("la_retention", "la_retention_with_state"):
    getattr(lib, _name).argtypes = [_vp, _vp, _vp, _fp, _fp, ctypes.POINTER(_f), _i, _i, _i, _i, _i, _i, _vp]
    getattr(lib, _name).restype = _i
lib.la_decode_step.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _i, _i, _i, _i, _f, _i, _vp]
lib.la_retention_decode_step.argtypes = [_vp, _vp, _vp, _fp, _fp, ctypes.POINTER(_f), _i, _i, _i, _i, _i, _vp]
lib.la_retention_decode_step.restype = _i
lib.la_causal_backward.argtypes = [_vp] * 13 + [_i, _i, _i, _i, _i, _f, _i, _vp]
lib.la_causal_backward.restype = _i
lib.la_favor_features.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]
lib.la_favor_features.restype = _i
lib.la_decode_step.restype = _i
lib.la_status_string.argtypes = [_i]
lib.la_status_string.restype = ctypes.c_char_p
lib.la_version.argtypes = []
lib.la_version.restype = _i
lib.la_device_status.argtypes = [_vp]
lib.la_device_status.restype = _i
lib.la_last_error_detail.argtypes = []
lib.la_last_error_detail.restype = ctypes.c_char_p
lib.la_kernel_launches.argtypes = []
lib.la_kernel_launches.restype = ctypes.c_ulonglong
lib.la_diag_force_segments.argtypes = [_i]
lib.la_diag_force_segments.restype = _i
lib.la_test_inject_missing_load.argtypes = [_i, ctypes.c_uint]
lib.la_test_inject_missing_load.restype = _i
lib.la_profile_enable.argtypes = [_i]
lib.la_profile_enable.restype = _i
lib.la_profile_read.argtypes = [_i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
lib.la_profile_read.restype = _i

# la_kernel ids of the device-time diagnostics
KERNELS = {"causal_main": 0, "causal_state": 1, "exact_head": 2, "causal_simt": 3, "global_state": 4,
           "global_read": 5, "decode": 6, "retention_main": 7, "retention_state": 8, "retention_decode": 9,
           "backward": 10, "favor": 11, "global_fused": 12}


class LinAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        detail = f"; {lib.la_last_error_detail().decode()}" if code in (4, 5, 7) else ""
        super().__init__(f"{fn}: {STATUS_NAMES.get(code, code)} ({status_string(code)}{detail})")


def status_string(code: int) -> str:
    return lib.la_status_string(code).decode()


def version() -> int:
    return lib.la_version()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"q, k, v must be float32 or bfloat16, got {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_in(q, k, v, nd):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != nd:
            raise ValueError(f"{name} must be a contiguous {nd}-d CUDA tensor")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share one dtype")
    if q.shape != k.shape or q.shape[:-1] != v.shape[:-1]:
        raise ValueError("q, k must have equal shapes and v the same leading dims")


def _state(S, z, lead, dk, dv, dev):
    if S is None:
        S = torch.empty(*lead, dk, dv, dtype=torch.float32, device=dev)
    if z is None:
        z = torch.empty(*lead, dk, dtype=torch.float32, device=dev)
    if S.dtype != torch.float32 or z.dtype != torch.float32 or not S.is_contiguous() or not z.is_contiguous():
        raise ValueError("S and z must be contiguous float32 tensors")
    if tuple(S.shape) != (*lead, dk, dv) or tuple(z.shape) != (*lead, dk):
        raise ValueError(f"S must be {(*lead, dk, dv)} and z {(*lead, dk)}")
    return S, z


def _seq_call(fn, q, k, v, out, S, z, eps, stream, need_state_in=False):
    _check_in(q, k, v, 4)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if need_state_in and (S is None or z is None):
        raise ValueError(f"{fn} needs the initial state S, z")
    S, z = _state(S, z, (B, H), dk, dv, q.device)
    if out is None:
        out = torch.empty(B, H, N, dv, dtype=torch.float32, device=q.device)
    if out.dtype != torch.float32 or not out.is_contiguous() or tuple(out.shape) != (B, H, N, dv):
        raise ValueError("out must be a contiguous float32 [B, H, N, d_v] tensor")
    rc = getattr(lib, fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z), B, H, N, dk, dv, float(eps),
                          _dt(q), _stream(stream))
    if rc != 0:
        raise LinAttnError(fn, rc)
    return out, S, z


def la_global(q, k, v, out=None, S=None, z=None, eps: float = 1e-6, stream=None):
    """Global read; returns (out, S, z).  S, z are overwritten with the whole-sequence state."""
    return _seq_call("la_global", q, k, v, out, S, z, eps, stream)


def la_causal(q, k, v, out=None, S=None, z=None, eps: float = 1e-6, stream=None):
    """Causal prefill from the zero state; returns (out, S, z) with the final state."""
    return _seq_call("la_causal", q, k, v, out, S, z, eps, stream)


def la_causal_noalloc(q, k, v, out=None, S=None, z=None, eps: float = 1e-6, stream=None):
    """la_causal without device allocation inside the library (fixed scratch; see linattn.h).

    Pass preallocated out, S, z to keep the whole call allocation-free: the
    binding only allocates the outputs that were not supplied.
    """
    return _seq_call("la_causal_noalloc", q, k, v, out, S, z, eps, stream)


def la_causal_features(phi_q, phi_k, v, out=None, S=None, z=None, eps: float = 1e-6, stream=None):
    """Causal prefill on given (non-negative) features; returns (out, S, z)."""
    return _seq_call("la_causal_features", phi_q, phi_k, v, out, S, z, eps, stream)


def la_global_features(phi_q, phi_k, v, out=None, S=None, z=None, eps: float = 1e-6, stream=None):
    """Global read on given (non-negative) features; returns (out, S, z)."""
    return _seq_call("la_global_features", phi_q, phi_k, v, out, S, z, eps, stream)


def la_favor_features(x, W, out=None, stream=None):
    """Positive random features of x [B, H, N, d] for projections W [m, d]: [B, H, N, m], x's dtype."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 4:
        raise ValueError("x must be a contiguous 4-d CUDA tensor")
    if not W.is_cuda or not W.is_contiguous() or W.dim() != 2 or W.shape[1] != x.shape[-1] or W.dtype != x.dtype:
        raise ValueError("W must be a contiguous [m, d] CUDA tensor of x's dtype")
    B, H, N, d = x.shape
    m = W.shape[0]
    if out is None:
        out = torch.empty(B, H, N, m, dtype=x.dtype, device=x.device)
    if out.dtype != x.dtype or not out.is_contiguous() or tuple(out.shape) != (B, H, N, m):
        raise ValueError("out must be a contiguous [B, H, N, m] tensor of x's dtype")
    rc = lib.la_favor_features(_ptr(x), _ptr(W), _ptr(out), B, H, N, d, m, _dt(x), _stream(stream))
    if rc != 0:
        raise LinAttnError("la_favor_features", rc)
    return out


def la_causal_with_state(q, k, v, S, z, out=None, eps: float = 1e-6, stream=None):
    """Causal prefill continuing from (S, z), which are updated in place; returns (out, S, z)."""
    return _seq_call("la_causal_with_state", q, k, v, out, S, z, eps, stream, need_state_in=True)


def _retention_call(fn, q, k, v, gamma, out, S, stream, need_state_in=False):
    _check_in(q, k, v, 4)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    g = [float(x) for x in gamma]
    if len(g) != H:
        raise ValueError(f"gamma must hold one decay per head ({H}), got {len(g)}")
    if need_state_in and S is None:
        raise ValueError(f"{fn} needs the initial state S")
    if S is None:
        S = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    if S.dtype != torch.float32 or not S.is_contiguous() or tuple(S.shape) != (B, H, dk, dv):
        raise ValueError(f"S must be a contiguous float32 {(B, H, dk, dv)} tensor")
    if out is None:
        out = torch.empty(B, H, N, dv, dtype=torch.float32, device=q.device)
    if out.dtype != torch.float32 or not out.is_contiguous() or tuple(out.shape) != (B, H, N, dv):
        raise ValueError("out must be a contiguous float32 [B, H, N, d_v] tensor")
    garr = (_f * max(H, 1))(*g)
    rc = getattr(lib, fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), garr, B, H, N, dk, dv, _dt(q),
                          _stream(stream))
    if rc != 0:
        raise LinAttnError(fn, rc)
    return out, S


def la_retention(q, k, v, gamma, out=None, S=None, stream=None):
    """Retention from the zero state (decay gamma[h] per head, no denominator); returns (out, S)."""
    return _retention_call("la_retention", q, k, v, gamma, out, S, stream)


def la_retention_with_state(q, k, v, S, gamma, out=None, stream=None):
    """Retention continuing from S, which is updated in place; returns (out, S)."""
    return _retention_call("la_retention_with_state", q, k, v, gamma, out, S, stream, need_state_in=True)


def la_decode_step(q, k, v, S, z, out=None, eps: float = 1e-6, stream=None):
    """One decode step; q, k [B, H, d_k], v [B, H, d_v]; S, z updated in place; returns out."""
    _check_in(q, k, v, 3)
    B, H, dk = q.shape
    dv = v.shape[-1]
    S, z = _state(S, z, (B, H), dk, dv, q.device)
    if out is None:
        out = torch.empty(B, H, dv, dtype=torch.float32, device=q.device)
    rc = lib.la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z), B, H, dk, dv, float(eps),
                            _dt(q), _stream(stream))
    if rc != 0:
        raise LinAttnError("la_decode_step", rc)
    return out


def la_retention_decode_step(q, k, v, S, gamma, out=None, stream=None):
    """One retention step; q, k [B, H, d_k], v [B, H, d_v]; S updated in place; returns out."""
    _check_in(q, k, v, 3)
    B, H, dk = q.shape
    dv = v.shape[-1]
    g = [float(x) for x in gamma]
    if len(g) != H:
        raise ValueError(f"gamma must hold one decay per head ({H}), got {len(g)}")
    if S is None or S.dtype != torch.float32 or not S.is_contiguous() or tuple(S.shape) != (B, H, dk, dv):
        raise ValueError(f"S must be a contiguous float32 {(B, H, dk, dv)} tensor")
    if out is None:
        out = torch.empty(B, H, dv, dtype=torch.float32, device=q.device)
    rc = lib.la_retention_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), (_f * max(H, 1))(*g), B, H,
                                      dk, dv, _dt(q), _stream(stream))
    if rc != 0:
        raise LinAttnError("la_retention_decode_step", rc)
    return out


def la_causal_backward(q, k, v, dout, S0=None, z0=None, dS=None, dz=None, need_state_grad: bool = False,
                       eps: float = 1e-6, stream=None):
    """Gradients of la_causal (la_causal_with_state when S0, z0 are given) for the
    upstream gradient ``dout`` of its output and, optionally, ``dS``, ``dz`` of its
    final state.  Returns (dq, dk, dv), plus (dS0, dz0) when ``need_state_grad``."""
    _check_in(q, k, v, 4)
    B, H, N, dk = q.shape
    dv = v.shape[-1]

    def f32(t, shape, name):
        if t is None:
            return None
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {shape}")
        return t

    dout = f32(dout, (B, H, N, dv), "dout")
    S0, dS = f32(S0, (B, H, dk, dv), "S0"), f32(dS, (B, H, dk, dv), "dS")
    z0, dz = f32(z0, (B, H, dk), "z0"), f32(dz, (B, H, dk), "dz")
    new = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=q.device)
    dq, dkk, dvv = new(B, H, N, dk), new(B, H, N, dk), new(B, H, N, dv)
    dS0, dz0 = (new(B, H, dk, dv), new(B, H, dk)) if need_state_grad else (None, None)
    rc = lib.la_causal_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(S0), _ptr(z0), _ptr(dS), _ptr(dz),
                                _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dS0), _ptr(dz0), B, H, N, dk, dv, float(eps),
                                _dt(q), _stream(stream))
    if rc != 0:
        raise LinAttnError("la_causal_backward", rc)
    return (dq, dkk, dvv, dS0, dz0) if need_state_grad else (dq, dkk, dvv)


def device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status: 0 = OK, 6 = a bounded wait timed out."""
    return int(lib.la_device_status(_stream(stream)))


def diag_force_segments(segments: int) -> None:
    """Diagnostics: segments per head of the tensor-core causal passes (0: the planner's choice)."""
    rc = lib.la_diag_force_segments(int(segments))
    if rc != 0:
        raise LinAttnError("la_diag_force_segments", rc)


def test_inject_missing_load(chunk: int, wait_us: int) -> None:
    """Testing only: the next tensor-core causal launch leaves out one key load of its
    first CTA and gives every wait ``wait_us`` microseconds (see linattn.h)."""
    rc = lib.la_test_inject_missing_load(int(chunk), int(wait_us))
    if rc != 0:
        raise LinAttnError("la_test_inject_missing_load", rc)


def profile_enable(on: bool = True) -> None:
    """Start (clearing the totals) or stop per-launch device timing."""
    lib.la_profile_enable(1 if on else 0)


def profile_read(kernel: str):
    """(total milliseconds, timed launches) of one kernel since profile_enable(True)."""
    ms, n = ctypes.c_double(), ctypes.c_longlong()
    rc = lib.la_profile_read(KERNELS[kernel], ctypes.byref(ms), ctypes.byref(n))
    if rc != 0:
        raise LinAttnError("la_profile_read", rc)
    return ms.value, n.value


def kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib.la_kernel_launches())
