"""Python access to the CPU oracle (``oracle.c``) plus the pages' closed-form costs.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
bench's CPU-baseline leg, never by the CUDA library or its binding.  Arrays are
numpy: bf16 data travels as ``uint16`` bit patterns, fp32 as ``float32``.

Closed forms below follow the page "AllGather" (tier6-model interconnect
notes), sections "理论下界" (eqs. ag-delay-lb, allgather-recv,
allgather-bw-lower-bound), "Ring AllGather" (eqs. ring-ag, ag-bidir-ring) and
"Recursive Doubling AllGather" (eqs. ag-recursive-doubling-full, rd-ag).
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

BF16, F32 = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i32, i64, vp, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
        L.orc_bf16_to_f32.restype = f32
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [f32]
        L.orc_bf16_to_f32_array.argtypes = [vp, vp, i64]
        L.orc_f32_to_bf16_array.argtypes = [vp, vp, i64]
        L.orc_reduce_rows.argtypes = [i32, i32, vp, i64, i64, i32, i32, vp]
        L.orc_owner_map.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        L.orc_flush.argtypes = [i32, i32, vp, i64, i32, vp, vp, vp, vp, i32, i32, vp, i32, i32, vp]
        L.orc_flush_probe.argtypes = [i32, i32, vp, vp, vp, i32, vp, i32, vp]
        L.orc_flush_partitioned.argtypes = [i32, i32, vp, i64, i32, vp, vp, vp, vp, i64, i32, vp, i32, vp]
        L.orc_bucket_relayout.argtypes = [i32, i32, vp, i64, i32, vp, vp, vp, vp, i64, i64, vp, i64, vp]
        L.orc_accumulate.argtypes = [i32, i64, vp, i32, vp, i32, i32, f32, vp]
        L.orc_accumulator_save.argtypes = [i32, i64, vp, vp]
        L.orc_accumulator_restore.argtypes = [i32, i64, vp, vp]
        L.orc_reduce_each_microbatch.argtypes = [i32, i32, i64, i32, vp, f32, vp]
        L.orc_reduce_scatter.argtypes = [i32, i64, i32, vp, i32, vp, i32]
        L.orc_allgather.argtypes = [i32, i64, i32, vp, vp, i32]
        L.orc_ring_allgather_steps.argtypes = [i32, vp, vp]
        L.orc_rd_allgather_steps.argtypes = [i32, vp, vp, vp, vp, vp]
        L.orc_bidir_ring_allgather_steps.argtypes = [i32, vp, vp]
        _lib = L
    return _lib


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle arrays are uint16 (bf16 bits) or float32, got {a.dtype}")


def _np_dtype(dt: int):
    return np.uint16 if dt == BF16 else np.float32


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments ({rc})")


# ------------------------------------------------------------------ bf16 ---

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    lib().orc_bf16_to_f32_array(b.ctypes.data, out.ctypes.data, b.size)
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(f.ctypes.data, out.ctypes.data, f.size)
    return out


# ------------------------------------------------------------- reduction ---

def reduce_rows(x: np.ndarray, pre_div: bool = True, out_dt: int | None = None) -> np.ndarray:
    """Reduce a [W, m] array over its rows (element rule of the bucket flush)."""
    x = np.ascontiguousarray(x)
    in_dt = _dt(x)
    out_dt = in_dt if out_dt is None else out_dt
    W, m = x.shape
    out = np.empty(m, dtype=_np_dtype(out_dt))
    _check(lib().orc_reduce_rows(W, in_dt, x.ctypes.data, m, m, int(pre_div), out_dt, out.ctypes.data), "reduce_rows")
    return out


def owner_map(world: int, groups, reduce_to_owner: bool = True, rank: int = 0) -> dict:
    """groups: list of (comm_ranks, numel array).  Returns per-parameter arrays
    (concatenated over groups) and the owned/total counts."""
    comm_size = np.array([len(g[0]) for g in groups], dtype=np.int32)
    comm_ranks = np.ascontiguousarray(np.concatenate([np.asarray(g[0], dtype=np.int32) for g in groups])
                                      if groups else np.zeros(0, np.int32), dtype=np.int32)
    n_params = np.array([len(g[1]) for g in groups], dtype=np.int32)
    numel = np.ascontiguousarray(np.concatenate([np.asarray(g[1], dtype=np.int64) for g in groups])
                                 if groups else np.zeros(0, np.int64), dtype=np.int64)
    P = int(n_params.sum())
    owner = np.empty(P, np.int32)
    lo = np.empty(P, np.int32)
    hi = np.empty(P, np.int32)
    n_owned = ctypes.c_int32()
    n_total = ctypes.c_int32()
    _check(lib().orc_owner_map(world, rank, len(groups), comm_size.ctypes.data, comm_ranks.ctypes.data,
                               n_params.ctypes.data, numel.ctypes.data, int(reduce_to_owner), owner.ctypes.data,
                               lo.ctypes.data, hi.ctypes.data, ctypes.byref(n_owned), ctypes.byref(n_total)),
           "owner_map")
    return {"owner": owner, "holder_lo": lo, "holder_hi": hi, "n_owned": n_owned.value, "n_total": n_total.value}


def flush(world: int, grads: np.ndarray, tasks: np.ndarray, owner: np.ndarray | None, n_params: int,
          dst: list | None, out_dt: int, pre_div: bool = True, reduce_to_owner: bool = True) -> dict:
    """Bucket flush.  grads: [W, ld] (modified in place when dst is None).
    tasks: structured array with param_id/offset/numel.  dst: list over ranks of
    lists over tasks of numpy arrays (or None for an empty buffer)."""
    assert grads.flags.c_contiguous
    in_dt = _dt(grads)
    W, ld = grads.shape
    assert W == world
    n_tasks = len(tasks)
    tp = np.ascontiguousarray(tasks["param_id"], dtype=np.int32)
    to = np.ascontiguousarray(tasks["offset"], dtype=np.int64)
    tn = np.ascontiguousarray(tasks["numel"], dtype=np.int64)
    own = None if owner is None else np.ascontiguousarray(owner, dtype=np.int32)
    table = None
    if dst is not None:
        table = (ctypes.c_void_p * max(world * n_tasks, 1))()
        for r in range(world):
            for t in range(n_tasks):
                buf = dst[r][t]
                if buf is not None:
                    assert buf.flags.c_contiguous and buf.dtype == _np_dtype(out_dt) and buf.size >= tn[t]
                    table[r * n_tasks + t] = buf.ctypes.data
    probe = np.zeros(4 + world, dtype=np.int64)
    _check(lib().orc_flush(world, in_dt, grads.ctypes.data, ld, n_tasks, tp.ctypes.data, to.ctypes.data,
                           tn.ctypes.data, None if own is None else own.ctypes.data, n_params, out_dt,
                           table, int(pre_div), int(reduce_to_owner), probe.ctypes.data), "flush")
    return _probe_dict(probe)


def _probe_dict(probe: np.ndarray) -> dict:
    return {"tasks": int(probe[0]), "reduced_elems": int(probe[1]), "owner_tasks": int(probe[2]),
            "owner_elems": int(probe[3]), "kept_elems": [int(v) for v in probe[4:]]}


def flush_probe(world: int, tasks: np.ndarray, owner: np.ndarray | None, n_params: int,
                has_dst: np.ndarray | None, reduce_to_owner: bool = True) -> dict:
    """Probe counters from metadata: has_dst is a [W, n_tasks] bool mask (None = in place)."""
    tp = np.ascontiguousarray(tasks["param_id"], dtype=np.int32)
    tn = np.ascontiguousarray(tasks["numel"], dtype=np.int64)
    own = None if owner is None else np.ascontiguousarray(owner, dtype=np.int32)
    has = None if has_dst is None else np.ascontiguousarray(has_dst, dtype=np.uint8)
    probe = np.zeros(4 + world, dtype=np.int64)
    _check(lib().orc_flush_probe(world, len(tasks), tp.ctypes.data, tn.ctypes.data,
                                 None if own is None else own.ctypes.data, n_params,
                                 None if has is None else has.ctypes.data, int(reduce_to_owner), probe.ctypes.data),
           "flush_probe")
    return _probe_dict(probe)


def flush_partitioned(world: int, grads: np.ndarray, tasks: np.ndarray, flat_offset: np.ndarray, part_size: int,
                      part_dst: list, out_dt: int, pre_div: bool = True) -> dict:
    """Every rank receives its partition's slice of the reduced bucket
    (part_dst[r]: numpy array of part_size elements, or None)."""
    assert grads.flags.c_contiguous
    W, ld = grads.shape
    tp = np.ascontiguousarray(tasks["param_id"], dtype=np.int32)
    to = np.ascontiguousarray(tasks["offset"], dtype=np.int64)
    tn = np.ascontiguousarray(tasks["numel"], dtype=np.int64)
    fo = np.ascontiguousarray(flat_offset, dtype=np.int64)
    table = (ctypes.c_void_p * world)()
    for r in range(world):
        if part_dst[r] is not None:
            assert part_dst[r].dtype == _np_dtype(out_dt) and part_dst[r].size >= part_size
            table[r] = part_dst[r].ctypes.data
    probe = np.zeros(4 + world, dtype=np.int64)
    _check(lib().orc_flush_partitioned(world, _dt(grads), grads.ctypes.data, ld, len(tasks), tp.ctypes.data,
                                       to.ctypes.data, tn.ctypes.data, fo.ctypes.data, part_size, out_dt, table,
                                       int(pre_div), probe.ctypes.data), "flush_partitioned")
    return _probe_dict(probe)


def bucket_relayout(grads: np.ndarray, tasks: np.ndarray, flat_offset: np.ndarray, part_size: int, seg: int,
                    out: np.ndarray) -> np.ndarray:
    """Rank-major relayout of a bucket into out ([W, >= W*seg]); returns seg_used."""
    assert grads.flags.c_contiguous and out.flags.c_contiguous and out.dtype == grads.dtype
    W, ld = grads.shape
    tp = np.ascontiguousarray(tasks["param_id"], dtype=np.int32)
    to = np.ascontiguousarray(tasks["offset"], dtype=np.int64)
    tn = np.ascontiguousarray(tasks["numel"], dtype=np.int64)
    fo = np.ascontiguousarray(flat_offset, dtype=np.int64)
    used = np.zeros(W, np.int64)
    _check(lib().orc_bucket_relayout(W, grads.dtype.itemsize, grads.ctypes.data, ld, len(tasks), tp.ctypes.data,
                                     to.ctypes.data, tn.ctypes.data, fo.ctypes.data, part_size, seg, out.ctypes.data,
                                     out.shape[1], used.ctypes.data), "bucket_relayout")
    return used


def accumulate(acc: np.ndarray, g: np.ndarray, first: bool, finalize: bool, scale: float = 1.0):
    """acc: [W, n] float32 (updated unless finalize); g: [W, n] bf16 bits or f32.
    Returns total [n] when finalize."""
    assert acc.dtype == np.float32 and acc.flags.c_contiguous and g.flags.c_contiguous and acc.shape == g.shape
    W, n = acc.shape
    total = np.empty(n, np.float32) if finalize else None
    _check(lib().orc_accumulate(W, n, acc.ctypes.data, _dt(g), g.ctypes.data, int(first), int(finalize), scale,
                                None if total is None else total.ctypes.data), "accumulate")
    return total


def accumulator_save(acc: np.ndarray) -> np.ndarray:
    """The reduced total a checkpoint holds: sum over replicas in rank order."""
    assert acc.dtype == np.float32 and acc.flags.c_contiguous
    W, n = acc.shape
    total = np.empty(n, np.float32)
    _check(lib().orc_accumulator_save(W, n, acc.ctypes.data, total.ctypes.data), "accumulator_save")
    return total


def accumulator_restore(total: np.ndarray, world: int) -> np.ndarray:
    """The unreduced form of a total: replica 0 holds it, the others hold zero."""
    t = np.ascontiguousarray(total, dtype=np.float32)
    acc = np.empty((world, len(t)), np.float32)
    _check(lib().orc_accumulator_restore(world, len(t), acc.ctypes.data, t.ctypes.data), "accumulator_restore")
    return acc


def reduce_each_microbatch(g: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """g: [M, W, n]; the per-micro-batch all-reduce then the sum over micro-batches."""
    g = np.ascontiguousarray(g)
    M, W, n = g.shape
    out = np.empty(n, np.float32)
    _check(lib().orc_reduce_each_microbatch(W, M, n, _dt(g), g.ctypes.data, scale, out.ctypes.data), "per-microbatch")
    return out


def reduce_scatter(x: np.ndarray, pre_div: bool = False, out_dt: int | None = None) -> np.ndarray:
    x = np.ascontiguousarray(x)
    N, M = x.shape
    in_dt = _dt(x)
    out_dt = in_dt if out_dt is None else out_dt
    if M % N:
        raise ValueError("M % N != 0")
    out = np.empty((N, M // N), dtype=_np_dtype(out_dt))
    _check(lib().orc_reduce_scatter(N, M, in_dt, x.ctypes.data, out_dt, out.ctypes.data, int(pre_div)),
           "reduce_scatter")
    return out


def allgather(x: np.ndarray, order: int = 0) -> np.ndarray:
    x = np.ascontiguousarray(x)
    N, S = x.shape
    out = np.empty((N, N * S), dtype=x.dtype)
    _check(lib().orc_allgather(N, S, x.dtype.itemsize, x.ctypes.data, out.ctypes.data, order), "allgather")
    return out


def ring_steps(n: int) -> dict:
    hold = np.empty((n, n, n), np.int32)
    recv = np.empty(n, np.int64)
    _check(lib().orc_ring_allgather_steps(n, hold.ctypes.data, recv.ctypes.data), "ring steps")
    return {"hold": hold, "recv_chunks": recv}


def rd_steps(n: int) -> dict:
    steps = max(1, int(round(math.log2(n)))) if n > 1 else 0
    partner = np.empty((max(steps, 1), n), np.int32)
    xfer = np.empty(max(steps, 1), np.int64)
    held = np.empty(max(steps, 1), np.int64)
    final = np.empty((n, n), np.int32)
    recv = np.empty(n, np.int64)
    _check(lib().orc_rd_allgather_steps(n, partner.ctypes.data, xfer.ctypes.data, held.ctypes.data,
                                        final.ctypes.data, recv.ctypes.data), "recursive doubling steps")
    return {"partner": partner[:steps], "xfer_chunks": xfer[:steps], "held_chunks": held[:steps],
            "final": final, "recv_chunks": recv}


def bidir_ring_steps(n: int) -> dict:
    steps = n // 2
    hold = np.empty((steps + 1, n, n), np.int32)
    recv = np.empty(n, np.int64)
    rc = lib().orc_bidir_ring_allgather_steps(n, hold.ctypes.data, recv.ctypes.data)
    if rc < 0:
        raise ValueError(f"bidirectional ring simulation failed ({rc})")
    return {"steps": rc, "hold": hold, "recv_chunks": recv}


# ----------------------------------------------------------- closed forms ---

def ag_latency_lower_bound(N: int, alpha: float) -> float:
    """eq. ag-delay-lb: ceil(log2 N) * alpha."""
    return math.ceil(math.log2(N)) * alpha if N > 1 else 0.0


def ag_recv(N: int, M: float) -> float:
    """eq. allgather-recv: each node must receive (N-1)/N * M."""
    return (N - 1) / N * M


def ag_bw_lower_bound(N: int, M: float, d: int, beta: float) -> float:
    """eq. allgather-bw-lower-bound: (N-1) M / (N d beta)."""
    return (N - 1) * M / (N * d * beta)


def ring_ag_time(N: int, M: float, alpha: float, beta: float) -> float:
    """eq. ring-ag: (N-1) (alpha + (M/N)/beta)."""
    return (N - 1) * (alpha + (M / N) / beta)


def bidir_ring_ag_time(N: int, M: float, alpha: float, beta: float) -> float:
    """eq. ag-bidir-ring: ceil((N-1)/2) (alpha + (M/N)/beta)."""
    return math.ceil((N - 1) / 2) * (alpha + (M / N) / beta)


def rd_ag_time(N: int, M: float, alpha: float, beta: float) -> float:
    """eq. ag-recursive-doubling-full: sum over steps j=1..log2 N of alpha + M 2^(j-1)/(N beta)."""
    steps = int(round(math.log2(N)))
    if 2 ** steps != N:
        raise ValueError("recursive doubling needs N = 2^k")
    return sum(alpha + M * 2 ** (j - 1) / (N * beta) for j in range(1, steps + 1))
