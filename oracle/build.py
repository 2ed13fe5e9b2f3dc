"""Compiles the FP64 CPU oracle (test infrastructure) into a shared library.

Plain gcc, no vendor toolchain: the oracle must run wherever the tests run.
``-ffp-contract=off`` keeps the compiler from fusing multiply-adds, so the oracle gives
the same bits on x86_64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rmsnorm_oracle.c")
LIB = os.path.join(HERE, "librmsnorm_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Builds ``librmsnorm_oracle.so`` next to the source if missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
