"""Parameter trees and bucket layouts of the synthetic workloads.

These are inputs to the bucket flush: which parameters exist, in which order
their gradients arrive, and how the arrival-order stream is cut into reduce
buckets.  The sizes and orders follow the workloads that the DeepSpeed issue
"DeepCompile ZeRO-1: reduce-to-owner instead of AllReduce" (section
"Additional context": 402.8M parameters, 806 MB of bf16 gradients; probe line:
52,428,800-element buckets) and the MaxText PR "Defer the data-parallel
gradient all-reduce to update() under gradient accumulation" (section
"Results": qwen3-0.6b) measure on.  Readings where the pages are silent:

* 402.8M tree: tied 98304x1024 embedding, 24 layers of
  [ln1.w, ln1.b, q, k, v, o (1024x1024 each), ln2.w, ln2.b, fc1 (1024x4096),
  fc2 (4096x1024)], final LayerNorm (w, b): 243 tensors, 402,753,536 elements.
* qwen3-0.6b tree: tied 151936x1024 embedding, 28 layers of [input norm,
  q 1024x2048, q_norm 128, k 1024x1024, k_norm 128, v 1024x1024, o 2048x1024,
  post-attention norm, gate/up 1024x3072, down 3072x1024], final norm:
  596,049,920 elements.
* Gradients arrive in reverse model order (backward).  Buckets are packed
  greedily in arrival order: a bucket is closed before a parameter that would
  overflow the capacity, and a parameter larger than the capacity gets a bucket
  of its own.  Within a bucket, tasks sit back to back in arrival order.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BUCKET_CAPACITY = 52_428_800  # elements, the bucket of the printed probe line

TASK_DTYPE = np.dtype([("param_id", "<i4"), ("pad", "<i4"), ("offset", "<i8"), ("numel", "<i8")])


@dataclass
class Tree:
    names: list[str]
    numel: np.ndarray  # int64, model (flat) order

    @property
    def total(self) -> int:
        return int(self.numel.sum())

    @property
    def n_params(self) -> int:
        return len(self.names)


def tree_402m() -> Tree:
    h, f, vocab, layers = 1024, 4096, 98304, 24
    names, sizes = ["embed"], [vocab * h]
    for i in range(layers):
        for n, s in (("ln1.w", h), ("ln1.b", h), ("q", h * h), ("k", h * h), ("v", h * h), ("o", h * h),
                     ("ln2.w", h), ("ln2.b", h), ("fc1", h * f), ("fc2", f * h)):
            names.append(f"l{i}.{n}")
            sizes.append(s)
    names += ["ln_f.w", "ln_f.b"]
    sizes += [h, h]
    return Tree(names, np.array(sizes, dtype=np.int64))


def tree_qwen3_06b() -> Tree:
    h, hq, hkv, hd, ffn, vocab, layers = 1024, 2048, 1024, 128, 3072, 151936, 28
    names, sizes = ["embed"], [vocab * h]
    for i in range(layers):
        for n, s in (("input_norm", h), ("q", h * hq), ("q_norm", hd), ("k", h * hkv), ("k_norm", hd),
                     ("v", h * hkv), ("o", hq * h), ("post_norm", h), ("gate", h * ffn), ("up", h * ffn),
                     ("down", ffn * h)):
            names.append(f"l{i}.{n}")
            sizes.append(s)
    names.append("norm")
    sizes.append(h)
    return Tree(names, np.array(sizes, dtype=np.int64))


def tree_tiny(seed: int = 1, count: int = 16) -> Tree:
    """``count`` parameters with sizes uniform in [1, 4096] (seeded)."""
    from . import int_sizes
    sizes = int_sizes(count, seed=seed, stream=0, lo=1, span=4096)
    return Tree([f"p{i}" for i in range(count)], sizes.astype(np.int64))


@dataclass
class Bucket:
    start: int           # element offset of the bucket in the arrival-order row
    size: int            # elements per replica row
    tasks: np.ndarray    # TASK_DTYPE, arrival order, offsets relative to ``start``


@dataclass
class Layout:
    """Arrival-order gradient row: param p occupies [row_offset[p], row_offset[p] + numel[p])."""
    tree: Tree
    arrival: np.ndarray        # param ids in arrival order
    row_offset: np.ndarray     # int64 per param id
    buckets: list[Bucket] = field(default_factory=list)

    @property
    def row_len(self) -> int:
        return self.tree.total


def arrival_layout(tree: Tree, capacity: int | None = BUCKET_CAPACITY, arrival: np.ndarray | None = None) -> Layout:
    """Lay the gradients out in arrival order (default: reverse model order) and pack buckets."""
    if arrival is None:
        arrival = np.arange(tree.n_params - 1, -1, -1, dtype=np.int64)
    row_offset = np.zeros(tree.n_params, dtype=np.int64)
    pos = 0
    for p in arrival:
        row_offset[p] = pos
        pos += int(tree.numel[p])
    cap = capacity if capacity is not None else max(pos, 1)
    buckets: list[Bucket] = []
    cur: list[int] = []
    cur_size = 0

    def close():
        nonlocal cur, cur_size
        if cur:
            start = int(row_offset[cur[0]])
            t = np.zeros(len(cur), dtype=TASK_DTYPE)
            t["param_id"] = cur
            t["offset"] = [int(row_offset[p]) - start for p in cur]
            t["numel"] = [int(tree.numel[p]) for p in cur]
            buckets.append(Bucket(start, cur_size, t))
        cur, cur_size = [], 0

    for p in arrival:
        n = int(tree.numel[p])
        if n > cap:
            close()
            cur, cur_size = [int(p)], n
            close()
            continue
        if cur_size + n > cap:
            close()
        cur.append(int(p))
        cur_size += n
    close()
    return Layout(tree, np.asarray(arrival, dtype=np.int64), row_offset, buckets)


def straddle_tree(world: int, bucket_elems: int, straddlers: int, pieces: int = 3) -> Tree:
    """A parameter group of ``bucket_elems`` elements cut so that exactly ``straddlers``
    of the W-1 interior partition boundaries (partition size ceil(T/W)) fall strictly
    inside a parameter; every other boundary falls between two parameters."""
    assert 0 <= straddlers <= world - 1 and bucket_elems >= world * pieces * 2
    part = -(-bucket_elems // world)
    bounds = [min(j * part, bucket_elems) for j in range(world + 1)]
    cuts: set[int] = set()
    for j in range(world):
        lo, hi = bounds[j], bounds[j + 1]
        for k in range(1, pieces):
            c = lo + (hi - lo) * k // pieces
            if lo < c < hi:
                cuts.add(c)
    for j in range(1, world):
        if bounds[j] < bucket_elems:
            cuts.add(bounds[j])
    for j in range(1, straddlers + 1):
        cuts.discard(bounds[j])
    edges = [0] + sorted(cuts) + [bucket_elems]
    sizes = [b - a for a, b in zip(edges[:-1], edges[1:]) if b > a]
    return Tree([f"s{i}" for i in range(len(sizes))], np.array(sizes, dtype=np.int64))
