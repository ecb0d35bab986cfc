"""Compile libdpred.so (the C-ABI library and its sm_103a kernels) in-tree.

Translation units compile in parallel with nvcc, then link into one shared
library next to this file.  --fmad=false and the explicit round-to-nearest
intrinsics in the kernels keep every fp32 operation a separate IEEE step.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sysconfig

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libdpred.so")
OBJDIR = os.path.join(HERE, "_build")
# The checked build (device-side bounds tests on every flush-kernel access,
# failures recorded as DPRED_E_BOUNDS) is a separate library, built on demand.
LIB_CHECKED = os.path.join(HERE, "libdpred_checked.so")
OBJDIR_CHECKED = os.path.join(HERE, "_build_checked")
FLUSH_UNITS = [f"flush_w{w}.cu" for w in (*(str(w) for w in range(2, 17)), "gen", "gen32", "genx")]
SOURCES = ["abi.cu", "flush_dispatch.cu", *FLUSH_UNITS, "accumulate.cu", "allgather.cu", "noalloc.cu", "selftest.cu",
           "relayout.cu", "schedule.cu", "owner_map.cu", "executor.cu", "ceiling.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", *ARCH, "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "-I", CSRC]


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dpred.h")]
    return [f for f in files if f.endswith((".cu", ".cuh", ".h"))]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps() + [os.path.abspath(__file__)])


def _compile(src: str, extra: list[str], objdir: str = OBJDIR) -> str:
    obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
    cmd = ["nvcc", *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


# The optional CPython call path for prepared flushes (argument marshalling
# only; see csrc/fastcall.c).  Built with the host C compiler when the Python
# headers are present; without them the binding uses ctypes for the same call.
FASTCALL = os.path.join(HERE, "_fastcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_fastcall(force: bool = False) -> str | None:
    """Compile the fast-call module; returns its path, or None when this
    Python has no headers or no C compiler (never raises)."""
    src = os.path.join(CSRC, "fastcall.c")
    deps = [src, os.path.join(INCLUDE, "dpred.h"), os.path.abspath(__file__)]
    if not force and os.path.exists(FASTCALL) and all(os.path.getmtime(d) <= os.path.getmtime(FASTCALL) for d in deps):
        return FASTCALL
    inc = sysconfig.get_paths().get("include") or ""
    if not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    cc = os.environ.get("CC", "cc")
    tmp = FASTCALL + ".tmp"
    try:
        r = subprocess.run([cc, "-O2", "-shared", "-fPIC", "-std=c11", "-Wall", "-I", inc, "-I", INCLUDE, src, "-o",
                            tmp], capture_output=True, text=True)
    except OSError:
        return None
    if r.returncode != 0:
        return None
    os.replace(tmp, FASTCALL)
    return FASTCALL


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    lib, objdir = (LIB_CHECKED, OBJDIR_CHECKED) if checked else (LIB, OBJDIR)
    if not checked:
        build_fastcall(force)
    if not force and not stale(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checked:
        extra.append("-DDPRED_CHECKED=1")
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, objdir), SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run(["nvcc", *ARCH, "-shared", *objs, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
