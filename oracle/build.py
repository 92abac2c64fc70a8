"""Compile the fp64 C oracle into ``oracle/liblaoracle.so`` (test infrastructure).

Flags keep IEEE double semantics on both x86_64 and aarch64: no fast-math and
no floating-point contraction into fused multiply-adds.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "liblaoracle.so")


def build_oracle() -> str:
    src = os.path.join(_HERE, "la_oracle.c")
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle())
