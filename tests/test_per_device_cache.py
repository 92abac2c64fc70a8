"""The per-device table behind the library's shared-memory opt-ins (CPU only).

CUDA function attributes belong to one device's context, so every launcher
records them per device.  This builds tests/native/per_device_cache_test.cpp
against the library's csrc/per_device.h with the host compiler and runs it.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_linear_attention_attn_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "per_device_cache_test.cpp")


def test_per_device_cache_keys_by_device(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "per_device_cache_test"
    subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, SRC, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"


def test_no_launcher_caches_device_state_process_wide():
    """No launcher keeps a process-wide once-flag for a device attribute: the only
    std::call_once left in the library is the driver entry-point lookup."""
    hits = []
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(CSRC, name)) as f:
            for i, line in enumerate(f, 1):
                if "call_once" in line or "once_flag" in line:
                    hits.append(f"{name}:{i}")
    assert len(hits) == 2 and all(h.startswith("causal_tc.cu:") for h in hits), hits
