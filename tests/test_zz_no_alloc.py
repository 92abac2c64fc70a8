"""la_causal_noalloc: the causal prefill entry point that allocates no device memory.

Some callers cannot let a library allocate device memory while they run: a
serving runtime that reserves all of its memory at start-up and forbids any
allocation after warm-up, or a process whose other framework already holds
nearly all device memory in its caching allocator.  For them the library keeps
the scratch that la_causal would allocate per call (the partial states of long
sequences split into segments) in one fixed device array instead.

These tests call the allocation-free entry point through the C ABI on two
calls in a row and check its outputs and final state against la_causal's and
against the fp64 oracle on sampled heads, within the parity tolerance used for
bf16 inputs.  The second call reuses the fixed array, which still holds the
first call's partial states.  The shapes are chosen so that both calls split
their heads into segments and use the array.  A third test watches the
device's stream-ordered memory pool and its free memory around the call: the
pool's high-water mark rises under la_causal (which allocates its scratch
there) and does not move under la_causal_noalloc.  The file is named so that
pytest collects it last.
"""
import ctypes

import pytest
import torch

import oracle
from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
# two shapes that split every head into segments (so the fixed array is used)
SHAPES = [(1, 2, 3000), (2, 3, 2500)]
SAMPLED_HEADS = {(1, 2, 3000): [0, 1], (2, 3, 2500): [0, 4]}

# CUmemPool_attribute values from cuda.h
CU_MEMPOOL_ATTR_USED_MEM_CURRENT = 7
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


class PoolWatch:
    """The current device's stream-ordered memory pool, read through the driver API."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetMemPool(ctypes.byref(self.pool), dev) == 0

    def _get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        zero = ctypes.c_uint64(0)  # resets the high-water mark to the current use
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(zero)) == 0

    def used(self):
        return self._get(CU_MEMPOOL_ATTR_USED_MEM_CURRENT)

    def high(self):
        return self._get(CU_MEMPOOL_ATTR_USED_MEM_HIGH)


def _inputs(w, B, H, N):
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    return (q, k, v), tuple(t.to(DEV) for t in (q, k, v))


def _check_against_oracle(w, host, got, shape):
    B, H, N = shape
    heads = SAMPLED_HEADS[shape]
    sel = lambda t: t.reshape(B * H, *t.shape[2:])[heads]
    q, k, v = (sel(t) for t in host)
    ro, rS, rz = oracle.causal(f64(q), f64(k), f64(v), eps=w.eps, nthreads=len(heads))
    out, S, z = (sel(t) for t in got)
    tau = TAU[w.torch_dtype]
    assert_close(out, ro, tau, f"out vs oracle {shape}")
    assert_close(S, rS, tau, f"S vs oracle {shape}")
    assert_close(z, rz, tau, f"z vs oracle {shape}")


def test_noalloc_matches_la_causal_and_oracle_on_two_calls_in_a_row(cuda_lib):
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    tau = TAU[w.torch_dtype]
    for B, H, N in SHAPES:
        host, (q, k, v) = _inputs(w, B, H, N)
        ref_out, ref_S, ref_z = L.la_causal(q, k, v, eps=w.eps)
        out, S, z = _nan(B, H, N, w.dv), _nan(B, H, w.dk, w.dv), _nan(B, H, w.dk)
        L.la_causal_noalloc(q, k, v, out=out, S=S, z=z, eps=w.eps)
        torch.cuda.synchronize()
        assert_close(out, f64(ref_out), tau, f"out {B}x{H}x{N}")
        assert_close(S, f64(ref_S), tau, f"S {B}x{H}x{N}")
        assert_close(z, f64(ref_z), tau, f"z {B}x{H}x{N}")
        _check_against_oracle(w, host, (out, S, z), (B, H, N))
    assert L.device_status() == 0


def test_noalloc_allocates_nothing(cuda_lib):
    """The pool's high-water mark rises under la_causal and stays put under
    la_causal_noalloc; device free memory is unchanged by the call."""
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    B, H, N = SHAPES[1]
    host, (q, k, v) = _inputs(w, B, H, N)
    out, S, z = _nan(B, H, N, w.dv), _nan(B, H, w.dk, w.dv), _nan(B, H, w.dk)
    # warm-up: the first call on the device looks up the fixed array's address (and loads
    # the kernels); it is made before anything is measured
    L.la_causal_noalloc(q, k, v, out=out, S=S, z=z, eps=w.eps)
    torch.cuda.synchronize()
    pool = PoolWatch()
    # positive control: la_causal takes its scratch from this pool
    pool.reset_high()
    base = pool.used()
    L.la_causal(q, k, v, eps=w.eps)
    torch.cuda.synchronize()
    assert pool.high() > base, "la_causal's scratch did not show in the pool (the probe sees nothing)"
    # the allocation-free call: no growth of the pool, no change of device free memory
    torch.cuda.synchronize()
    pool.reset_high()
    base = pool.used()
    free0, _ = torch.cuda.mem_get_info()
    L.la_causal_noalloc(q, k, v, out=out, S=S, z=z, eps=w.eps)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert pool.high() == base, f"pool high-water {pool.high()} > {base}: la_causal_noalloc allocated"
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across la_causal_noalloc"
    _check_against_oracle(w, host, (out, S, z), (B, H, N))
    assert L.device_status() == 0


def test_noalloc_small_and_float32_shapes_need_no_scratch(cuda_lib):
    """Shapes that take a single segment (or the fp32 path) also match la_causal."""
    L = cuda_lib
    for name, (B, H, N) in [("causal_bf16", (1, 1, 100)), ("causal_f32_small", (1, 2, 256))]:
        w = inputs.WORKLOADS[name]
        q, k, v = (t.to(DEV) for t in inputs.make_qkv(w, N=N, B=B, H=H))
        ref_out, ref_S, ref_z = L.la_causal(q, k, v, eps=w.eps)
        out, S, z = L.la_causal_noalloc(q, k, v, eps=w.eps)
        torch.cuda.synchronize()
        tau = TAU[w.torch_dtype]
        assert_close(out, f64(ref_out), tau, "out")
        assert_close(S, f64(ref_S), tau, "S")
