"""Helpers for the GPU parity tests: device tensors filled by the shared
generator, bit views, and the oracle side of a flush built from the oracle's
own owner map (no reduction arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

import datagen
import oracle
from tests.helpers import holder_sets, oracle_dst

TORCH_DT = {datagen.BF16: torch.bfloat16, datagen.F32: torch.float32}


def device_matrix(rows, cols, dt, kind, seed, stream0=0, col0=0, sigma=1.0, ld=None, extra=0):
    """A CUDA tensor [rows, ld] filled in columns [0, cols) (ld defaults to cols)."""
    ld = cols if ld is None else ld
    t = torch.empty(rows * ld + extra, dtype=TORCH_DT[dt], device="cuda")
    datagen.fill_device(t.data_ptr(), rows, cols, ld, dt, kind, seed, stream0, 1, col0, sigma,
                        torch.cuda.current_stream().cuda_stream)
    return t[: rows * ld].view(rows, ld)


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a CUDA tensor's bit patterns (uint16 for bf16, uint32 for fp32)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def np_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


def oracle_flush(world, grads_host, tasks, tree_numel, groups, out_dt, pre_div, rto, n_params):
    """Run the oracle flush with destinations derived from the oracle's own
    owner map.  Returns (dst lists, oracle owner map, probe)."""
    om = oracle.owner_map(world, groups, rto)
    holders = holder_sets(om["holder_lo"], om["holder_hi"])
    dst = oracle_dst(world, tasks, holders, out_dt == datagen.BF16)
    probe = oracle.flush(world, grads_host.copy(), tasks, om["owner"], n_params, dst, out_dt, pre_div, rto)
    return dst, om, probe
