"""alpha-beta cost model of the AllGather schedules.

Page "AllGather" (tier6-model interconnect notes): eq. ring-ag (N-1 steps of
alpha plus one chunk of M/N bytes), eq. ag-bidir-ring (ceil((N-1)/2) such
steps) and eq. rd-ag (log2 N steps whose payload doubles each step, total
(N-1)M/N).  `beta` is the per-node link bandwidth in bytes/s, M the gathered
bytes per node.  Used by the bench to compare measured step-by-step schedule
times with the model.
"""
from __future__ import annotations

import math


def ring(N: int, M: float, alpha: float, beta: float) -> float:
    steps = N - 1
    return steps * alpha + steps * (M / N) / beta


def bidirectional_ring(N: int, M: float, alpha: float, beta: float) -> float:
    steps = -(-(N - 1) // 2)
    return steps * alpha + steps * (M / N) / beta


def recursive_doubling(N: int, M: float, alpha: float, beta: float) -> float:
    k = N.bit_length() - 1
    if 1 << k != N:
        raise ValueError("recursive doubling needs N = 2^k")
    return k * alpha + sum((M / N) * (1 << j) for j in range(k)) / beta


def lower_bounds(N: int, M: float, alpha: float, beta: float, links: int = 1) -> tuple[float, float]:
    """Latency and bandwidth lower bounds: ceil(log2 N) alpha, (N-1) M / (N links beta)."""
    return math.ceil(math.log2(N)) * alpha if N > 1 else 0.0, (N - 1) * M / (N * links * beta)
