"""Seeded synthetic inputs shared by the tests, the bench and the CPU oracle's harness.

Values come from ``datagen.h`` (SplitMix64 in counter mode, Irwin-Hall normals,
uniform[-1, 1), bf16 by truncation) through ``libdatagen.so``; the same library
fills host memory (pthreads) and device memory (a CUDA kernel) with equal bits.
``workloads`` holds the parameter trees and bucket layouts of the synthetic
workloads.  Nothing in this package reduces, scales or rounds a gradient.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdatagen.so")

NORMAL, UNIFORM = 0, 1
BF16, F32 = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        from . import build as _build
        L = ctypes.CDLL(_build.build())
        i64, u64, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
        L.dg_normal_scale.restype = ctypes.c_float
        L.dg_normal_scale.argtypes = [ctypes.c_float]
        fill = [vp, ctypes.c_int, ctypes.c_int, i64, i64, i64, i64, u64, u64, u64, ctypes.c_float]
        L.dg_fill_device.argtypes = fill + [vp]
        L.dg_fill_host.argtypes = fill + [ctypes.c_int]
        L.dg_sample_host.argtypes = [vp, ctypes.c_int, ctypes.c_int, i64, vp, vp, u64, ctypes.c_float]
        L.dg_int_sizes.argtypes = [vp, i64, u64, u64, i64, i64]
        _lib = L
    return _lib


def normal_scale(sigma: float) -> float:
    """sigma * 2^-16 rounded to fp32, the multiplier of the Irwin-Hall recipe."""
    return float(lib().dg_normal_scale(sigma))


def _scale(kind: int, sigma: float) -> float:
    return normal_scale(sigma) if kind == NORMAL else 0.0


def fill_host(arr: np.ndarray, dtype: int, kind: int, seed: int, stream0: int = 0, stream_step: int = 1,
              col0: int = 0, sigma: float = 1.0, threads: int | None = None) -> np.ndarray:
    """Fill a C-contiguous 2-D host array (uint16 for bf16 bits, float32 for f32)."""
    assert arr.ndim == 2 and arr.flags.c_contiguous
    assert arr.dtype == (np.uint16 if dtype == BF16 else np.float32)
    rows, cols = arr.shape
    threads = threads or os.cpu_count() or 1
    rc = lib().dg_fill_host(arr.ctypes.data, dtype, kind, rows, cols, cols, col0, seed, stream0, stream_step,
                            _scale(kind, sigma), threads)
    if rc != 0:
        raise ValueError(f"dg_fill_host failed ({rc})")
    return arr


def host_matrix(rows: int, cols: int, dtype: int, kind: int, seed: int, stream0: int = 0, stream_step: int = 1,
                col0: int = 0, sigma: float = 1.0) -> np.ndarray:
    arr = np.empty((rows, cols), dtype=np.uint16 if dtype == BF16 else np.float32)
    return fill_host(arr, dtype, kind, seed, stream0, stream_step, col0, sigma)


def fill_device(ptr: int, rows: int, cols: int, ld: int, dtype: int, kind: int, seed: int, stream0: int = 0,
                stream_step: int = 1, col0: int = 0, sigma: float = 1.0, stream: int = 0) -> None:
    """Fill device memory at ``ptr`` ([rows, cols], row stride ``ld`` elements) on a CUDA stream."""
    rc = lib().dg_fill_device(ctypes.c_void_p(ptr), dtype, kind, rows, cols, ld, col0, seed, stream0, stream_step,
                              _scale(kind, sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"dg_fill_device failed ({rc})")


def sample_host(streams, idx, dtype: int, kind: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    """Values number ``idx[j]`` of stream ``streams[j]``, one by one."""
    s = np.ascontiguousarray(streams, dtype=np.uint64)
    i = np.ascontiguousarray(idx, dtype=np.int64)
    assert s.shape == i.shape and s.ndim == 1
    out = np.empty(s.shape, dtype=np.uint16 if dtype == BF16 else np.float32)
    rc = lib().dg_sample_host(out.ctypes.data, dtype, kind, len(s), s.ctypes.data, i.ctypes.data, seed,
                              _scale(kind, sigma))
    if rc != 0:
        raise ValueError(f"dg_sample_host failed ({rc})")
    return out


def int_sizes(count: int, seed: int, stream: int = 0, lo: int = 1, span: int = 4096) -> np.ndarray:
    """``count`` integers uniform in [lo, lo + span), e.g. parameter sizes."""
    out = np.empty(count, dtype=np.int64)
    rc = lib().dg_int_sizes(out.ctypes.data, count, seed, stream, lo, span)
    if rc != 0:
        raise ValueError("dg_int_sizes failed")
    return out


def stream_id(replica: int, microbatch: int = 0) -> int:
    """Stream number of one replica row of one micro-batch."""
    return (microbatch << 16) | replica
