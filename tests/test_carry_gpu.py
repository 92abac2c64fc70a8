"""The carry of the causal prefill across segments, at every segment count.

The tensor-core path cuts each head into G segments: G = 1 carries the state
through all chunks in one CTA; G > 1 starts each segment from the sum of the
first pass's pieces over the earlier ones ("Linear Attention: From Pairwise
Reads to a Recurrent State", "A recurrence need not force token-serial
training").  la_diag_force_segments fixes G so that both carries can be timed;
every G must give the oracle's result within the bf16 bar.
"""
import pytest
import torch

import oracle
from causal_linear_attention_attn_gb300 import inputs
from paritylib import TAU, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("G", [1, 2, 3, 7, 0])
def test_every_segment_count_matches_the_oracle(cuda_lib, G):
    L = cuda_lib
    w = inputs.WORKLOADS["causal_bf16"]
    B, H, N = 1, 2, 2000  # 16 chunks per head
    q, k, v = inputs.make_qkv(w, N=N, B=B, H=H)
    S0 = torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(2))
    z0 = torch.rand(B, H, 128, generator=torch.Generator().manual_seed(3)) * 50 + 1
    try:
        L.diag_force_segments(G)
        out, S, z = L.la_causal(q.to(DEV), k.to(DEV), v.to(DEV), eps=w.eps)
        Sc, zc = S0.to(DEV), z0.to(DEV)
        out2, _, _ = L.la_causal_with_state(q.to(DEV), k.to(DEV), v.to(DEV), Sc, zc, eps=w.eps)
        torch.cuda.synchronize()
    finally:
        L.diag_force_segments(0)
    assert L.device_status() == 0
    tau = TAU[w.torch_dtype]
    ro, rS, rz = oracle.causal(f64(q), f64(k), f64(v), eps=w.eps, nthreads=2)
    assert_close(out, ro, tau, f"out G={G}")
    assert_close(S, rS, tau, f"S G={G}")
    assert_close(z, rz, tau, f"z G={G}")
    ro2, rS2, rz2 = oracle.causal(f64(q), f64(k), f64(v), eps=w.eps, S0=f64(S0), z0=f64(z0), nthreads=2)
    assert_close(out2, ro2, tau, f"out from state G={G}")
    assert_close(Sc, rS2, tau, f"S from state G={G}")
