"""A second, independent restatement of the flush element rule in numpy fp32.

Used only on tiny inputs to cross-check the C oracle: numpy's float32 division
and addition are IEEE round-to-nearest operations, and bf16 rounding is done by
PyTorch's CPU cast (round to nearest even), not by the oracle's bit arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def reduce_f32(x: np.ndarray, pre_div: bool, order=None) -> np.ndarray:
    """x: [W, m] float32 -> [m] float32, summed in `order` (default 0..W-1)."""
    W = x.shape[0]
    order = list(range(W)) if order is None else list(order)
    wf = np.float32(W)
    y = None
    for r in order:
        t = (x[r] / wf).astype(np.float32) if pre_div else x[r].astype(np.float32)
        y = t.copy() if y is None else (y + t).astype(np.float32)
    return y


def flush(world, grads_f32, tasks, owner, reduce_to_owner, pre_div, out_bf16, holders):
    """Returns {(rank, param_id): values} for every delivered, non-empty destination.
    holders[p] = set of ranks with a real buffer for p."""
    out = {}
    for t in tasks:
        pid, off, n = int(t["param_id"]), int(t["offset"]), int(t["numel"])
        y = reduce_f32(grads_f32[:, off:off + n], pre_div)
        vals = f32_to_bf16_bits(y) if out_bf16 else y
        root = owner[pid] if (reduce_to_owner and owner is not None and owner[pid] >= 0) else -1
        for r in range(world):
            if (root < 0 or root == r) and r in holders[pid]:
                out[(r, pid)] = vals
    return out
