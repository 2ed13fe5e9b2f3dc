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
LN_SRC = os.path.join(HERE, "layernorm_oracle.c")
LN_LIB = os.path.join(HERE, "liblayernorm_oracle.so")


def compile_c(src: str, lib: str) -> str:
    """gcc -shared of one oracle source, FP contraction off."""
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def _build(src: str, lib: str, force: bool) -> str:
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(src):
        return lib
    return compile_c(src, lib)


def build_oracle(force: bool = False) -> str:
    """Builds ``librmsnorm_oracle.so`` next to the source if missing or stale."""
    return _build(SRC, LIB, force)


def build_layernorm_oracle(force: bool = False) -> str:
    """Builds ``liblayernorm_oracle.so`` next to the source if missing or stale."""
    return _build(LN_SRC, LN_LIB, force)


if __name__ == "__main__":
    print(build_oracle(force=True))
    print(build_layernorm_oracle(force=True))
