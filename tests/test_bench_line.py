"""The bench line's layout on CPU: every form is compact, and the forms a log that
keeps only the line's end must show (the long-context causal form, the global form
and the decode step) come last."""
import json

import bench


def _form(name, kernel, **extra):
    res = {"workload": name, "ms_per_call": 1.2345678, "tokens_per_s": 3.58e9, "gpu_launches": 9,
           "roofline": {"kernel": kernel, "ms_per_launch": 0.86873, "frac": 0.9112, "traffic": 634838016},
           "step_roofline": {"frac": 0.6767}, "clocks": {"sm_mhz": 2070.0, "reasons": []}}
    res.update(extra)
    return res


def test_forms_end_with_the_configs_a_tail_must_show():
    names = ["causal_bf16_long", "global_bf16", "causal_bf16_with_state", "retention_bf16", "favor_bf16",
             "causal_bf16_backward", "decode_bf16", "retention_decode_bf16"]
    forms = {n: _form(n, "k") for n in names}
    forms["causal_bf16_backward"]["tensor_roofline"] = {"frac": 0.0607}
    forms["decode_bf16"]["gbs"] = 6866.3
    out = bench.ordered_forms(forms)
    assert list(out)[-3:] == ["decode_bf16", "global_bf16", "causal_bf16_long"]
    assert set(out) == set(names)
    # a headline of realistic size in front: the last 1500 characters still hold those three forms
    line = json.dumps({"metric": "m" * 120, "config": {"x": "y" * 400}, "roofline": {"r": "z" * 300},
                       "e2e": {"e": "w" * 150}, "cpu_baseline": {"c": "v" * 150}, "forms": out})
    tail = line[-1500:]
    for n in ("decode_bf16", "global_bf16", "causal_bf16_long"):
        assert n in tail


def test_compact_keeps_the_figures_and_drops_the_rest():
    c = bench.compact(_form("causal_bf16_long", "causal_main"))
    assert c == {"ms": 1.23457, "tokens_per_s": 3.58e9, "step_frac": 0.6767, "kernel": "causal_main",
                 "kernel_ms": 0.86873, "kernel_frac": 0.9112, "traffic": 634838016}
    throttled = _form("global_bf16", "global_state", clocks={"sm_mhz": 1500.0, "reasons": ["sw_power_cap"]})
    assert bench.compact(throttled)["clock_reasons"] == ["sw_power_cap"]


def test_one_pass_global_kernel_counts_the_whole_call_once():
    """The one-pass global kernel's algorithmic bytes are the call's: q, k, v read and out, S, z
    written once (640 B per token at d = 64 in bf16), the state not read back as the two-kernel
    form's read does."""
    from causal_linear_attention_attn_gb300 import inputs

    w = inputs.WORKLOADS["global_bf16"]
    fused = bench.kernel_bytes(w, "global_fused")
    assert fused == bench.seq_bytes(w)
    assert fused == w.BH * (w.N * 640 + (64 * 64 + 64) * 4)
    two = bench.kernel_bytes(w, "global_state") + bench.kernel_bytes(w, "global_read")
    assert two - fused == w.BH * (64 * 64 + 64) * 4
