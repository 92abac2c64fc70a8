"""The tensor-core feature map on every finite bf16 input.

The tensor-core kernels evaluate phi(x) = ELU(x) + 1 on packed bf16 pairs
without a branch: e^x from the hardware base-2 exponential in fp32, rounded
to bf16, and x + 1 as a bf16 add, combined by min and max.  The result should
be phi(x) correctly rounded to bf16 ("Linear Attention Math", "Feature maps:
elu+1"; "线性注意力从头到尾讲清楚" §8).

It is observed through la_global on one-token sequences (bf16, d = 128): the
normalizer z of a head is the sum over its tokens of phi(k) as the tensor-core
state build rounds it, so with one token z = bf16(phi(k_0)) exactly.  All
65,280 finite bf16 bit patterns are spread over 510 heads of 128 features and
compared with the oracle's fp64 phi rounded to bf16 (round to nearest even).
The hardware exponential flushes results below the smallest normal float
(x below about -87.34) to zero; there the kernel may return 0 where the
correctly rounded value is a subnormal below 1.2e-38.
"""
import numpy as np
import pytest
import torch

import oracle

DEV = "cuda"
D = 128


def _bf16_round(x):
    """Round float64 values to bf16 (8 significant bits, round half to even), subnormals included."""
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    a = np.abs(x[nz])
    _, e = np.frexp(a)  # a = m 2^e, m in [0.5, 1)
    quantum = np.exp2(np.maximum(e - 8, -133))  # bf16: 8 significant bits; subnormal quantum 2^-133
    out[nz] = np.sign(x[nz]) * np.round(a / quantum) * quantum  # np.round: half to even
    return out


def test_round_helper_against_torch_on_float32_values():
    """The rounding helper agrees with torch's float32 -> bf16 conversion (RNE)."""
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(100000, generator=g) * s for s in (1e-30, 1e-3, 1.0, 1e3, 1e30)])
    assert np.array_equal(_bf16_round(x.double().numpy()), x.to(torch.bfloat16).double().numpy())


@pytest.mark.gpu
def test_phi_on_every_finite_bf16_value(cuda_lib):
    L = cuda_lib
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    bits = bits[finite]
    assert bits.size == 65280 and bits.size % D == 0  # 256 patterns have the all-ones exponent
    heads = bits.size // D
    x = (bits << 16).view(np.float32).astype(np.float64)  # the bf16 values, exactly
    k = torch.from_numpy((bits << 16).view(np.float32).copy()).to(torch.bfloat16).reshape(1, heads, 1, D)
    assert np.array_equal(k.double().numpy().ravel(), x)
    q = torch.zeros_like(k)
    v = torch.zeros_like(k)  # S = 0, so the read cannot overflow
    _, _, z = L.la_global(q.to(DEV), k.to(DEV), v.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    got = z.double().cpu().numpy().ravel()
    want = _bf16_round(oracle.phi(x))
    tiny = oracle.phi(x) < 2.0 ** -126  # the exponential flushes results below the normal range
    exact = got == want
    assert np.all(exact | (tiny & (got == 0))), (
        f"{np.count_nonzero(~exact & ~tiny)} inputs differ, e.g. x = {x[~exact & ~tiny][:4]}: "
        f"got {got[~exact & ~tiny][:4]}, want {want[~exact & ~tiny][:4]}")
    assert np.all(exact[~tiny])
    assert L.device_status() == 0
