"""C-ABI host checks that need no GPU: exported symbols, status strings and
argument validation (every validation path returns before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest
import torch

from conftest import ROOT

L = pytest.importorskip("causal_linear_attention_attn_gb300.linattn")

OK, INVALID, UNSUPPORTED, MISALIGNED, NO_DEVICE = 0, 1, 2, 3, 7


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"LA_API\s+[\w\s\*]*?\b(la_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    names = _declared_symbols()
    for n in ("la_global", "la_causal", "la_causal_with_state", "la_causal_noalloc", "la_decode_step", "la_status_string",
              "la_version", "la_retention", "la_retention_with_state", "la_retention_decode_step",
              "la_causal_backward", "la_favor_features", "la_causal_features", "la_global_features"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in _declared_symbols():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings():
    assert L.version() >> 16 == 1
    for code in range(9):
        s = L.status_string(code)
        assert isinstance(s, str) and s
    assert L.status_string(99) == "unknown status"


# A fake, 16-byte aligned, non-NULL address: never dereferenced, because every
# call below fails validation (or has nothing to do) before touching the GPU.
P = 1 << 20


def seq(fn="la_causal", q=P, k=P, v=P, out=P, S=P, z=P, B=1, H=1, N=8, dk=32, dv=32, eps=1e-6, dt=1, stream=None):
    return getattr(L.lib, fn)(q, k, v, out, S, z, B, H, N, dk, dv, eps, dt, stream)


@pytest.mark.parametrize("fn", ["la_causal", "la_global", "la_causal_with_state", "la_causal_noalloc"])
def test_sequence_validation(fn):
    assert seq(fn, q=None) == INVALID
    assert seq(fn, v=None) == INVALID
    assert seq(fn, out=None) == INVALID
    assert seq(fn, S=None) == INVALID
    assert seq(fn, z=None) == INVALID
    assert seq(fn, B=-1) == INVALID
    assert seq(fn, N=-3) == INVALID
    assert seq(fn, dk=0) == INVALID
    assert seq(fn, eps=-1e-6) == INVALID
    assert seq(fn, eps=float("nan")) == INVALID
    assert seq(fn, eps=float("inf")) == INVALID
    assert seq(fn, dk=48) == UNSUPPORTED
    assert seq(fn, dv=256) == UNSUPPORTED
    assert seq(fn, dt=5) == UNSUPPORTED
    assert seq(fn, q=P + 8) == MISALIGNED
    assert seq(fn, out=P + 4) == MISALIGNED
    assert seq(fn, z=P + 2) == MISALIGNED
    # nothing to do: no heads
    assert seq(fn, B=0) == OK
    assert seq(fn, H=0, q=None, k=None, v=None, out=None, S=None, z=None) == OK
    # empty sequences still need the state buffers (they are written or kept)
    assert seq(fn, N=0, q=None, k=None, v=None, out=None, S=None) == INVALID


def test_decode_validation():
    f = L.lib.la_decode_step
    args = dict(q=P, k=P, v=P, out=P, S=P, z=P, B=2, H=2, dk=64, dv=64, eps=1e-6, dt=1, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["q"], a["k"], a["v"], a["out"], a["S"], a["z"], a["B"], a["H"], a["dk"], a["dv"], a["eps"],
                 a["dt"], a["stream"])

    assert call(k=None) == INVALID
    assert call(S=None) == INVALID
    assert call(H=-1) == INVALID
    assert call(eps=float("nan")) == INVALID
    assert call(dv=96) == UNSUPPORTED
    assert call(S=P + 4) == MISALIGNED
    assert call(B=0) == OK


def ret(fn="la_retention", q=P, k=P, v=P, out=P, S=P, gamma=(0.9,), B=1, H=1, N=8, dk=128, dv=128, dt=1,
        stream=None):
    g = None if gamma is None else (ctypes.c_float * max(len(gamma), 1))(*gamma)
    return getattr(L.lib, fn)(q, k, v, out, S, g, B, H, N, dk, dv, dt, stream)


@pytest.mark.parametrize("fn", ["la_retention", "la_retention_with_state"])
def test_retention_validation(fn):
    assert ret(fn, q=None) == INVALID
    assert ret(fn, out=None) == INVALID
    assert ret(fn, S=None) == INVALID
    assert ret(fn, gamma=None) == INVALID
    assert ret(fn, gamma=(float("nan"),)) == INVALID
    assert ret(fn, gamma=(float("inf"),)) == INVALID
    assert ret(fn, N=-1) == INVALID
    assert ret(fn, dk=0) == INVALID
    # outside every retention kernel (fp32, d in {32, 64, 128} and gamma in [0, 1] are served)
    assert ret(fn, dt=7) == UNSUPPORTED
    assert ret(fn, dk=48) == UNSUPPORTED
    assert ret(fn, dv=96) == UNSUPPORTED
    assert ret(fn, gamma=(1.01,)) == UNSUPPORTED
    assert ret(fn, gamma=(-0.01,)) == UNSUPPORTED
    assert ret(fn, H=2, gamma=(0.5, 1.5)) == UNSUPPORTED
    assert ret(fn, H=129, gamma=(0.9,) * 129) == UNSUPPORTED
    assert ret(fn, v=P + 8) == MISALIGNED
    assert ret(fn, S=P + 4) == MISALIGNED
    assert ret(fn, B=0) == OK
    assert ret(fn, H=0, gamma=None, q=None, k=None, v=None, out=None, S=None) == OK


def test_retention_decode_validation():
    f = L.lib.la_retention_decode_step

    def call(q=P, k=P, v=P, out=P, S=P, gamma=(0.9, 0.9), B=2, H=2, dk=64, dv=64, dt=1):
        g = None if gamma is None else (ctypes.c_float * max(len(gamma), 1))(*gamma)
        return f(q, k, v, out, S, g, B, H, dk, dv, dt, None)

    assert call(k=None) == INVALID
    assert call(S=None) == INVALID
    assert call(gamma=None) == INVALID
    assert call(gamma=(0.9, float("nan"))) == INVALID
    assert call(H=-1) == INVALID
    assert call(dv=96) == UNSUPPORTED
    assert call(dt=3) == UNSUPPORTED
    assert call(gamma=(0.9, -0.1)) == UNSUPPORTED
    assert call(gamma=(1.5, 0.9)) == UNSUPPORTED
    assert call(H=129, gamma=(0.9,) * 129) == UNSUPPORTED
    assert call(S=P + 4) == MISALIGNED
    assert call(B=0) == OK


def test_favor_validation():
    f = L.lib.la_favor_features

    def call(x=P, Wp=P, phi=P, B=1, H=2, N=8, d=128, m=128, dt=1):
        return f(x, Wp, phi, B, H, N, d, m, dt, None)

    assert call(x=None) == INVALID
    assert call(phi=None) == INVALID
    assert call(N=-1) == INVALID
    assert call(m=0) == INVALID
    assert call(m=96) == UNSUPPORTED
    assert call(m=512) == UNSUPPORTED  # m = 256 (m = 2d at d = 128) is the largest
    assert call(d=256) == UNSUPPORTED  # the input dimension stays a head size
    assert call(d=48) == UNSUPPORTED
    assert call(dt=4) == UNSUPPORTED
    assert call(Wp=P + 2) == MISALIGNED
    assert call(B=0) == OK
    assert call(N=0, x=None, Wp=None, phi=None) == OK
    assert seq("la_causal_features", q=None) == INVALID
    assert seq("la_causal_features", dk=48) == UNSUPPORTED
    assert seq("la_global_features", v=None) == INVALID
    assert seq("la_global_features", dv=96) == UNSUPPORTED
    # 256 given features only with d_v <= 128, and only on the calls that take given features
    assert seq("la_causal_features", dk=512) == UNSUPPORTED
    assert seq("la_global_features", dk=256, dv=256) == UNSUPPORTED
    assert seq("la_causal", dk=256) == UNSUPPORTED
    assert seq("la_global", dk=256) == UNSUPPORTED
    assert seq("la_causal_features", dk=256, S=P + 4) == MISALIGNED


def test_backward_validation():
    f = L.lib.la_causal_backward

    def call(q=P, k=P, v=P, dout=P, S0=None, z0=None, dS=None, dz=None, dq=P, dk=P, dv=P, dS0=None, dz0=None,
             B=1, H=2, N=8, d_k=64, d_v=64, eps=1e-6, dt=1):
        return f(q, k, v, dout, S0, z0, dS, dz, dq, dk, dv, dS0, dz0, B, H, N, d_k, d_v, eps, dt, None)

    assert call(dout=None) == INVALID
    assert call(dq=None) == INVALID
    assert call(v=None) == INVALID
    assert call(N=-1) == INVALID
    assert call(eps=float("nan")) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(d_k=48) == UNSUPPORTED
    assert call(dt=2) == UNSUPPORTED
    assert call(dS=P + 4) == MISALIGNED
    assert call(dz0=P + 8) == MISALIGNED
    assert call(B=0) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_device_reports_no_device():
    assert seq("la_causal") == NO_DEVICE
    assert seq("la_global") == NO_DEVICE
    assert ret("la_retention") == NO_DEVICE


def test_binding_rejects_bad_tensors_before_the_library():
    q = torch.zeros(1, 1, 4, 32)
    with pytest.raises(ValueError):
        L.la_causal(q, q, q)  # CPU tensors
    with pytest.raises(ValueError):
        L.la_decode_step(q, q, q, None, None)
    with pytest.raises(ValueError):
        L.la_retention(q, q, q, [0.9])
    qc = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        L.la_retention(qc, qc, qc, [0.9])  # CPU tensors; also one decay for two heads


def test_profile_diagnostics_without_launches():
    L.profile_enable(True)
    for name in L.KERNELS:
        assert L.profile_read(name) == (0.0, 0)
    L.profile_enable(False)
    ms, n = ctypes.c_double(), ctypes.c_longlong()
    assert L.lib.la_profile_read(len(L.KERNELS), ctypes.byref(ms), ctypes.byref(n)) == INVALID
    assert L.lib.la_profile_read(-1, ctypes.byref(ms), ctypes.byref(n)) == INVALID
    assert L.lib.la_profile_read(0, None, ctypes.byref(n)) == INVALID


def test_fault_injection_hook_validates_its_arguments():
    """Only invalid arguments here: a valid call would arm the one-shot injection for a
    later GPU test in the same process."""
    f = L.lib.la_test_inject_missing_load
    assert f(-1, 1000) == INVALID
    assert f(0, 0) == INVALID
    assert f(0, 1000001) == INVALID


def test_segment_override_validates_and_resets():
    f = L.lib.la_diag_force_segments
    assert f(-1) == INVALID and f(4097) == INVALID
    assert f(0) == OK  # the planner's choice (the default)
