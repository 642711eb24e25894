"""Builds the oracle's C library beside its source with gcc: liboracle.so
(single-threaded; the checker the tests use) and liboracle_omp.so (the same source with
-fopenmp: the CPU baseline, its independent rows spread over the host cores).

Plain C11, -O2, -ffp-contract=off (no fused multiply-add), no -ffast-math, no
architecture-specific flags: it gives the same results on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.c")
OUT = os.path.join(_HERE, "liboracle.so")
OUT_OMP = os.path.join(_HERE, "liboracle_omp.so")


def _build_one(out: str, extra, force: bool) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-ffp-contract=off", *extra,
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False, parallel: bool = False) -> str:
    """Path of the single-threaded library (parallel=False) or the OpenMP one; both are
    (re)built when missing or older than the source."""
    single = _build_one(OUT, [], force)
    omp = _build_one(OUT_OMP, ["-fopenmp"], force)
    return omp if parallel else single


if __name__ == "__main__":
    print(build(force=True), build(parallel=True))
