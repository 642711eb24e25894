"""Builds the oracle's C library (liboracle.so) beside its source with gcc.

Plain C11, -O2, -ffp-contract=off (no fused multiply-add), no -ffast-math, no
architecture-specific flags: it gives the same results on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.c")
OUT = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True))
