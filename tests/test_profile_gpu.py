"""Device-time diagnostics: every launch of a call is timed on its own stream."""
import pytest
import torch

DEV = "cuda"

pytestmark = pytest.mark.gpu


def test_profile_counts_and_times_each_kernel(cuda_lib):
    L = cuda_lib
    g = torch.Generator(device="cpu").manual_seed(5)
    q, k, v = (torch.randn(1, 2, 2000, 128, generator=g).div(128 ** 0.5).bfloat16().to(DEV) for _ in range(3))
    L.la_causal(q, k, v)  # warm-up (one-time attribute set-up)
    torch.cuda.synchronize()
    n0 = L.kernel_launches()
    L.profile_enable(True)
    for _ in range(3):
        L.la_causal(q, k, v)
    L.profile_enable(False)
    torch.cuda.synchronize()
    launched = L.kernel_launches() - n0
    counts = {name: L.profile_read(name) for name in L.KERNELS}
    assert sum(n for _, n in counts.values()) == launched
    ms, n = counts["causal_main"]
    assert n == 3 and 0 < ms < 1000
    assert counts["exact_head"][1] == 3
    L.la_causal(q, k, v)  # profiling off: nothing more is recorded
    assert L.profile_read("causal_main") == (ms, 3)

    S = torch.zeros(4, 2, 64, 64, device=DEV)
    z = torch.zeros(4, 2, 64, device=DEV)
    x = torch.randn(4, 2, 64, device=DEV)
    L.profile_enable(True)
    L.la_decode_step(x, x, x, S, z)
    torch.cuda.synchronize()
    assert L.profile_read("decode")[1] == 1
    assert L.profile_read("causal_main") == (0.0, 0)
    L.profile_enable(False)


def test_global_form_takes_one_pass_when_the_heads_fill_the_sms(cuda_lib):
    """d = 64 with a head per SM: one kernel builds and reads each head; with few heads the
    state build and the read are two launches."""
    L = cuda_lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = torch.Generator(device="cpu").manual_seed(6)
    for heads, expect in ((sms, {"global_fused": 1}), (4, {"global_state": 1, "global_read": 1})):
        q, k, v = (torch.randn(1, heads, 300, 64, generator=g).div(8.0).bfloat16().to(DEV) for _ in range(3))
        L.la_global(q, k, v)  # warm-up (one-time attribute set-up)
        torch.cuda.synchronize()
        L.profile_enable(True)
        L.la_global(q, k, v)
        L.profile_enable(False)
        torch.cuda.synchronize()
        got = {name: L.profile_read(name)[1] for name in L.KERNELS}
        assert {name: n for name, n in got.items() if n} == expect
