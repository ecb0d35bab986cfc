"""Compile the CPU oracle (plain C) into oracle/liboracle.so.

Flags keep every fp32 operation a separate IEEE round-to-nearest step:
-fno-fast-math and -ffp-contract=off (GCC on aarch64 otherwise fuses a*b+c).
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def command() -> list[str]:
    return ["gcc", *CFLAGS, SRC, "-o", LIB + ".tmp", "-lm"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    subprocess.run(command(), check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
