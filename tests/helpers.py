"""Test-side helpers shared by the oracle and GPU test files (no reduction arithmetic)."""
from __future__ import annotations

import numpy as np

BF16_SENTINEL = np.uint16(0x7FC1)   # a NaN pattern no reduction of finite inputs produces
F32_SENTINEL_BITS = np.uint32(0x7FC00123)


def sentinel_array(n: int, out_bf16: bool) -> np.ndarray:
    if out_bf16:
        return np.full(n, BF16_SENTINEL, dtype=np.uint16)
    return np.full(n, F32_SENTINEL_BITS, dtype=np.uint32).view(np.float32)


def is_sentinel(a: np.ndarray, out_bf16: bool) -> np.ndarray:
    if out_bf16:
        return a.view(np.uint16) == BF16_SENTINEL
    return a.view(np.uint32) == F32_SENTINEL_BITS


def holder_sets(holder_lo, holder_hi) -> list[set]:
    return [set(range(lo, hi + 1)) if lo >= 0 else set() for lo, hi in zip(holder_lo, holder_hi)]


def oracle_dst(world: int, tasks, holders: list[set], out_bf16: bool):
    """Rank r gets a real buffer (pre-filled with the sentinel) for every task
    whose parameter it holds; None elsewhere (torch.empty([0]) in the issue)."""
    dst = [[None] * len(tasks) for _ in range(world)]
    for t, task in enumerate(tasks):
        pid, n = int(task["param_id"]), int(task["numel"])
        for r in holders[pid]:
            dst[r][t] = sentinel_array(n, out_bf16)
    return dst


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)
