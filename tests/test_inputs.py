"""Seeded input generators: determinism, per-head regeneration, shapes and scales."""
import math

import torch

from causal_linear_attention_attn_gb300 import inputs

W = inputs.WORKLOADS


def test_workloads_match_the_five_configurations_and_the_next_rows():
    assert [(w.B, w.H, w.N, w.dk, w.dv, w.dtype) for w in W.values()] == [
        (1, 2, 256, 32, 32, "f32"), (8, 16, 4096, 64, 64, "bf16"), (4, 16, 8192, 128, 128, "bf16"),
        (1, 32, 131072, 128, 128, "bf16"), (4, 16, 8192, 128, 128, "bf16"), (4, 16, 8192, 128, 128, "bf16"),
        (256, 32, 1, 128, 128, "bf16")]
    assert W["decode_bf16"].prefix == 1024 and W["decode_bf16"].steps == 1000
    assert all(w.eps == 1e-6 for w in W.values() if w.form != "retention")


def test_favor_projections():
    w = W["favor_bf16"]
    P = inputs.favor_projections(w)
    assert P.shape == (128, 128) and P.dtype == torch.bfloat16
    assert torch.equal(P, inputs.favor_projections(w))
    assert abs(P.float().std().item() - 1.0) < 0.05


def test_retention_gammas():
    g = inputs.retention_gamma(16)
    assert g[0] == 1 - 2 ** -5 and g[7] == 1 - 2 ** -12 and g[8:] == g[:8]
    # exact in float32, inside the supported range [0.75, 1)
    assert all(float(torch.tensor(x, dtype=torch.float32)) == x and 0.75 <= x < 1 for x in g)


def test_deterministic_and_per_head_reproducible():
    w = W["causal_bf16"]
    a = inputs.make_qkv(w, N=32, B=2, H=3)
    b = inputs.make_qkv(w, N=32, B=2, H=3)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q1, k1, v1 = inputs.make_qkv(w, N=32, heads=[4])
    assert torch.equal(q1[0], a[0][1, 1]) and torch.equal(v1[0], a[2][1, 1])


def test_scales_and_dtypes():
    w = W["causal_bf16"]
    q, k, v = inputs.make_qkv(w, N=4096, B=1, H=1)
    assert q.dtype == torch.bfloat16
    assert abs(q.float().std().item() - 1 / math.sqrt(128)) < 0.01
    assert abs(v.float().std().item() - 1.0) < 0.05
    q, _, _ = inputs.make_qkv(W["causal_f32_small"])
    assert q.dtype == torch.float32 and q.shape == (1, 2, 256, 32)


def test_decode_inputs():
    w = W["decode_bf16"]
    q, k, v = inputs.decode_step_qkv(w, 3, B=2, H=3)
    assert q.shape == (2, 3, 128) and v.dtype == torch.bfloat16
    q2, _, _ = inputs.decode_step_qkv(w, 3, B=2, H=3)
    assert torch.equal(q, q2)
    kp, vp = inputs.decode_prefix(w, heads=[0, 5])
    assert kp.shape == (2, 1024, 128)
    assert abs(kp.float().std().item() - 1.0) < 0.05
