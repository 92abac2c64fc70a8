"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait in the tensor-core causal pass is bounded.  A wait that
runs out raises the CTA's abort word and the device status word; the CTA
drains the copies and tensor-core work it has issued, frees its tensor memory
and exits, and la_device_status reports LA_ERR_TIMEOUT.  The test hook
la_test_inject_missing_load makes the next launch leave out one key load of
its first CTA (a barrier that nothing will complete) and shortens every wait
to one millisecond, on a two-chunk sequence.  The test checks the reported
status, then that the context is still usable: the next normal call matches
the fp64 oracle.
"""
import pytest
import torch

import oracle
from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
LA_ERR_TIMEOUT = 6


def test_missing_load_times_out_and_the_next_call_is_correct(cuda_lib):
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    B, H, N = 1, 1, 256  # one segment of two 128-token chunks
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    assert L.device_status() == 0
    L.test_inject_missing_load(1, 1000)  # chunk 1's keys never arrive; waits give up after 1 ms
    L.la_causal(qd, kd, vd, eps=w.eps)
    assert L.device_status() == LA_ERR_TIMEOUT
    assert L.device_status() == 0  # reading the status cleared it
    # the injection was one-shot and the context is usable: a normal call is correct
    out, S, z = L.la_causal(qd, kd, vd, eps=w.eps)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    ro, rS, rz = oracle.causal(f64(q), f64(k), f64(v), eps=w.eps)
    tau = TAU[w.torch_dtype]
    assert_close(out, ro, tau, "out")
    assert_close(S, rS, tau, "S")
    assert_close(z, rz, tau, "z")


def test_injection_for_a_chunk_past_the_end_changes_nothing(cuda_lib):
    """An armed chunk that the launch does not have leaves out no load."""
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=200, B=1, H=2)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    L.test_inject_missing_load(5, 1000)
    out, S, z = L.la_causal(qd, kd, vd, eps=w.eps)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    ro, rS, rz = oracle.causal(f64(q), f64(k), f64(v), eps=w.eps)
    assert_close(out, ro, TAU[w.torch_dtype], "out")
