"""la_causal_noalloc: the causal prefill entry point that allocates no device memory.

Some callers cannot let a library allocate device memory while they run: a
serving runtime that reserves all of its memory at start-up and forbids any
allocation after warm-up, or a process whose other framework already holds
nearly all device memory in its caching allocator.  For them the library keeps
the scratch that la_causal would allocate per call (the partial states of long
sequences split into segments) in one fixed device array instead.

These tests call the allocation-free entry point through the C ABI and check
its outputs and final state against la_causal's, within the parity tolerance
used for bf16 inputs, on two calls in a row: the second call reuses the fixed
array, which still holds the first call's partial states.  The shapes are
chosen so that both calls split their heads into segments and use the array.
The file is named so that pytest collects it last.
"""
import pytest
import torch

from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def test_noalloc_matches_la_causal_on_two_calls_in_a_row(cuda_lib):
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    for B, H, N in [(1, 2, 3000), (2, 3, 2500)]:
        q, k, v = (t.to(DEV) for t in inputs.make_qkv(w, N=N, B=B, H=H))
        ref_out, ref_S, ref_z = L.la_causal(q, k, v, eps=w.eps)
        out, S, z = _nan(B, H, N, w.dv), _nan(B, H, w.dk, w.dv), _nan(B, H, w.dk)
        L.la_causal_noalloc(q, k, v, out=out, S=S, z=z, eps=w.eps)
        torch.cuda.synchronize()
        tau = TAU[w.torch_dtype]
        assert_close(out, f64(ref_out), tau, f"out {B}x{H}x{N}")
        assert_close(S, f64(ref_S), tau, f"S {B}x{H}x{N}")
        assert_close(z, f64(ref_z), tau, f"z {B}x{H}x{N}")
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
