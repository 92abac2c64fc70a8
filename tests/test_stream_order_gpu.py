"""Work queued after a call on the same stream sees every output of it.

Each call runs its passes on the caller's stream, each allowed to start
beside its predecessor; the last one waits for the others before it
completes.  These tests consume the outputs with stream-ordered work only
(device copies queued right behind the call, no host synchronisation in
between) and compare the copies with the oracle."""
import dataclasses

import pytest
import torch

from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, oracle_seq

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("form,shape", [("causal", (2, 2, 3000, 128)), ("causal", (1, 3, 9000, 128)),
                                        ("global", (4, 8, 1500, 64)), ("global", (1, 2, 5000, 128)),
                                        ("global", (4, 40, 700, 64))])
def test_outputs_complete_for_the_next_work_on_the_stream(cuda_lib, form, shape):
    B, H, N, d = shape
    base = inputs.WORKLOADS["causal_bf16" if form == "causal" else "global_bf16"]
    w = dataclasses.replace(base, dk=d, dv=d)
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    fn = cuda_lib.la_causal if form == "causal" else cuda_lib.la_global
    with torch.cuda.stream(stream):
        # slow the stream down first so the call's kernels are still queued when the copies are enqueued
        ballast = torch.randn(4096, 4096, device=DEV)
        for _ in range(4):
            ballast = ballast @ ballast * 1e-3
        out, S, z = fn(qd, kd, vd, eps=w.eps, stream=stream)
        out_c, S_c, z_c = out.clone(), S.clone(), z.clone()  # stream-ordered reads of the results
        out.fill_(float("nan"))
        S.fill_(float("nan"))
        z.fill_(float("nan"))
    stream.synchronize()
    ro, rS, rz = oracle_seq(form, q, k, v, w.eps)
    tau = TAU[w.torch_dtype]
    assert_close(out_c, ro, tau, "out")
    assert_close(S_c, rS, tau, "S")
    assert_close(z_c, rz, tau, "z")
    assert cuda_lib.device_status() == 0


def test_back_to_back_calls_on_one_stream(cuda_lib):
    """A second call reusing the buffers of the first starts only after the first has finished."""
    w = inputs.WORKLOADS["causal_bf16"]
    q1, k1, v1 = (t.to(DEV) for t in inputs.make_qkv(w, N=4000, B=1, H=4))
    w2 = dataclasses.replace(w, seed=w.seed + 7)
    q2, k2, v2 = inputs.make_qkv(w2, N=4000, B=1, H=4)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        out, S, z = cuda_lib.la_causal(q1, k1, v1, eps=w.eps, stream=stream)
        first = out.clone()
        cuda_lib.la_causal(q2.to(DEV), k2.to(DEV), v2.to(DEV), out=out, S=S, z=z, eps=w.eps, stream=stream)
    stream.synchronize()
    r1, _, _ = oracle_seq("causal", *(t.cpu() for t in (q1, k1, v1)), w.eps)
    r2, rS2, rz2 = oracle_seq("causal", q2, k2, v2, w.eps)
    assert_close(first, r1, TAU[w.torch_dtype], "first call")
    assert_close(out, r2, TAU[w.torch_dtype], "second call")
    assert_close(S, rS2, TAU[w.torch_dtype], "S")
