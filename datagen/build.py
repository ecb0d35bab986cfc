"""Compile datagen.cu (host pthread fill + device fill kernel) into datagen/libdatagen.so."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "datagen.cu")
HDR = os.path.join(HERE, "datagen.h")
LIB = os.path.join(HERE, "libdatagen.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def command() -> list[str]:
    return ["nvcc", "-O3", *ARCH, "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-ffp-contract=off",
            SRC, "-o", LIB + ".tmp", "-lpthread"]


def stale() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(SRC), os.path.getmtime(HDR))


def build(force: bool = False) -> str:
    if force or stale():
        subprocess.run(command(), check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
