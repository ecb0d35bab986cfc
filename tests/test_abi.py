"""The C-ABI library without a GPU: it loads, exports every entry point its
header declares, and its host-only entry points (owner map, probe counters,
argument validation) agree with the oracle.  No call here launches a kernel:
the device entry points are only called with arguments they must reject."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import zero_collectives_gb300 as zc
from datagen import workloads
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from zero_collectives_gb300 import build
    build.build()
    return zc.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dpred.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dpred_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert zc.version().startswith("dpred")


def test_owner_map_matches_oracle_402m(L):
    tree = workloads.tree_402m()
    for rto in (True, False):
        got = zc.build_owner_map(8, [(None, tree.numel)], rto)
        ref = oracle.owner_map(8, [(list(range(8)), tree.numel)], rto)
        for k in ("owner", "holder_lo", "holder_hi"):
            assert np.array_equal(getattr(got, k), ref[k])
        assert (got.n_owned, got.n_total) == (ref["n_owned"], ref["n_total"])
    assert zc.build_owner_map(8, [(None, tree.numel)]).report() == \
        "DeepCompile reduce_to_owner: 236/243 gradients reduce to one rank"


def test_owner_map_matches_oracle_random_groups(L):
    rng = np.random.default_rng(12)
    for _ in range(300):
        world = int(rng.integers(1, 17))
        groups_o, groups_z = [], []
        for g in range(int(rng.integers(1, 4))):
            sizes = rng.integers(0, 5000, size=int(rng.integers(0, 30)))
            kind = rng.integers(0, 3)
            ranks = list(range(world))
            if kind == 1 and world > 1:
                ranks = list(range(max(1, world // 2)))
            elif kind == 2 and world > 1:
                ranks = ranks[::-1]
            groups_o.append((ranks, sizes))
            groups_z.append((ranks, sizes))
        rank = int(rng.integers(0, world))
        got = zc.build_owner_map(world, groups_z, True, rank)
        ref = oracle.owner_map(world, groups_o, True, rank)
        for k in ("owner", "holder_lo", "holder_hi"):
            assert np.array_equal(getattr(got, k), ref[k])
        assert (got.n_owned, got.n_total) == (ref["n_owned"], ref["n_total"])


def test_probe_counters_match_oracle(L):
    tree = workloads.tree_402m()
    om = zc.build_owner_map(8, [(None, tree.numel)])
    layout = workloads.arrival_layout(tree)
    for b in layout.buckets:
        n = len(b.tasks)
        ptrs = []
        has = np.zeros((8, n), bool)
        for r in range(8):
            for t in range(n):
                p = int(b.tasks["param_id"][t])
                held = om.holder_lo[p] <= r <= om.holder_hi[p]
                has[r, t] = held
                ptrs.append(0x1000 + 16 * (r * n + t) if held else 0)
        table = zc.DstTable(8, n, ptrs)
        for rto in (True, False):
            got = zc.flush_probe(8, b.tasks, om.owner, table, rto, flush_index=5)
            ref = oracle.flush_probe(8, b.tasks, om.owner, tree.n_params, has, rto)
            assert got.flush_index == 5
            assert (got.tasks, got.reduced_elems, got.owner_tasks, got.owner_elems) == \
                (ref["tasks"], ref["reduced_elems"], ref["owner_tasks"], ref["owner_elems"])
            assert got.kept_elems == ref["kept_elems"]
        inplace = zc.flush_probe(8, b.tasks, om.owner, None, True)
        ref = oracle.flush_probe(8, b.tasks, om.owner, tree.n_params, None, True)
        assert inplace.kept_elems == ref["kept_elems"]


def test_probe_line_reproduces_printed_line(golden_dir, L):
    meta, line = {}, None
    for raw in open(os.path.join(golden_dir, "probe_line.txt")):
        raw = raw.rstrip("\n")
        if raw.startswith("[dc-probe]"):
            line = raw
        elif raw and not raw.startswith("#"):
            k, v = raw.split("=")
            meta[k] = int(v)
    world = meta["world"]
    per = 52_428_800 // world
    sizes = []
    for j in range(world):
        k = 15 if j < 6 else 14
        base = per // k
        sizes += [base] * (k - 1) + [per - base * (k - 1)]
    tree = workloads.Tree([f"p{i}" for i in range(len(sizes))], np.array(sizes, np.int64))
    b = workloads.arrival_layout(tree, capacity=None).buckets[0]
    om = zc.build_owner_map(world, [(None, tree.numel)], reduce_to_owner=False)
    n = len(b.tasks)
    ptrs = [0x1000 if om.holder_lo[int(b.tasks["param_id"][t])] <= r <= om.holder_hi[int(b.tasks["param_id"][t])]
            else 0 for r in range(world) for t in range(n)]
    pr = zc.flush_probe(world, b.tasks, om.owner, zc.DstTable(world, n, ptrs), False, flush_index=meta["flush_index"])
    assert pr.line(meta["rank"], zc.BF16, True) == line
    # the same line straight from the C-ABI, and its argument checks
    raw = zc._Probe()
    L.dpred_flush_probe(world, b.tasks.ctypes.data, n, om.owner.ctypes.data, len(om.owner),
                        zc.DstTable(world, n, ptrs).c, 0, ctypes.byref(raw))
    raw.flush_index = meta["flush_index"]
    buf = ctypes.create_string_buffer(256)
    assert L.dpred_probe_format(ctypes.byref(raw), world, meta["rank"], zc.BF16, 1, buf, 256) == 0
    assert buf.value.decode() == line
    assert L.dpred_probe_format(ctypes.byref(raw), world, world, zc.BF16, 1, buf, 256) == -1   # rank out of range
    assert L.dpred_probe_format(ctypes.byref(raw), world, 0, 7, 1, buf, 256) == -1             # bad dtype
    small = ctypes.create_string_buffer(16)
    assert L.dpred_probe_format(ctypes.byref(raw), world, 0, zc.BF16, 1, small, 16) == -3      # too small
    log = []
    plog = zc.ProbeLog(rank=0, limit=20, sink=log.append)
    for i in range(25):
        pr.flush_index = plog.next_index()
        plog.record(pr, zc.BF16, True)
    assert len(log) == 20


def _tasks(spec):
    t = np.zeros(len(spec), dtype=zc.TASK_DTYPE)
    for i, (p, o, n) in enumerate(spec):
        t[i] = (p, 0, o, n)
    return t


def _call_flush(L, world=4, in_dt=0, grads=0x10000, ld=100, tasks=None, owner=None, n_params=0, out_dt=0,
                dst=None, checked=0):
    tasks = _tasks([(0, 0, 10)]) if tasks is None else tasks
    own = None if owner is None else np.ascontiguousarray(owner, np.int32)
    return L.dpred_flush_bucket(world, in_dt, grads, ld, tasks.ctypes.data, len(tasks),
                                None if own is None else own.ctypes.data, n_params if own is not None else 0,
                                out_dt, dst, 1, 1, checked, None, None, 0, None)


def test_validation_rejects_before_launch(L):
    E = {"INVAL": -1, "ALIGN": -2, "SIZE": -3, "MISMATCH": -4}
    assert _call_flush(L, world=0) == E["INVAL"]
    assert _call_flush(L, world=65) == E["INVAL"]
    assert _call_flush(L, in_dt=7) == E["INVAL"]
    assert _call_flush(L, ld=5) == E["SIZE"]                              # task outside the row
    assert _call_flush(L, grads=0x10001) == E["ALIGN"]                    # bf16 needs 2-byte alignment
    assert _call_flush(L, grads=0) == E["INVAL"]
    assert _call_flush(L, out_dt=1) == E["INVAL"]                         # in place needs equal dtypes
    assert _call_flush(L, tasks=_tasks([(0, 0, 10), (1, 5, 10)]), ld=100) == E["SIZE"]  # overlap in place
    assert _call_flush(L, tasks=_tasks([(3, 0, 10)]), owner=[0, 1], n_params=2) == E["INVAL"]
    assert _call_flush(L, tasks=_tasks([(0, 0, 10)]), owner=[9], n_params=1) == E["INVAL"]  # owner not a rank
    bad = _tasks([(0, -1, 10)])
    assert _call_flush(L, tasks=bad) == E["INVAL"]
    # checked mode: an owned task with a buffer on a non-owner rank
    tbl = (ctypes.c_void_p * 4)(0x20000, 0x30000, None, None)
    assert _call_flush(L, tasks=_tasks([(0, 0, 10)]), owner=[0], n_params=1, dst=tbl, checked=1) == E["MISMATCH"]
    assert b"owned by rank 0" in L.dpred_last_error()
    # reduce-scatter / allgather / accumulate argument checks
    assert L.dpred_reduce_scatter(4, 10, 0, 0x1000, 0, 0x2000, 0, None) == E["SIZE"]
    assert L.dpred_reduce_scatter(0, 8, 0, 0x1000, 0, 0x2000, 0, None) == E["INVAL"]
    assert L.dpred_allgather(4, 8, 0, 0x1000, 0x2000, 2, None) == E["INVAL"]
    assert L.dpred_allgather(4, 8, 0, 0x1001, 0x2000, 0, None) == E["ALIGN"]
    assert L.dpred_accumulate_microbatch(4, -1, 0x1000, 0, 0x2000, 1, 0, ctypes.c_float(1.0), None, None) == E["INVAL"]
    assert L.dpred_accumulate_microbatch(4, 8, 0x1000, 0, 0x2000, 1, 1, ctypes.c_float(1.0), None, None) == E["INVAL"]
    assert L.dpred_accumulate_microbatch(4, 8, 0x1002, 0, 0x2000, 1, 0, ctypes.c_float(1.0), None, None) == E["ALIGN"]


def test_empty_calls_are_no_ops(L):
    # zero tasks / zero elements enqueue nothing and succeed without a GPU
    t = np.zeros(0, dtype=zc.TASK_DTYPE)
    assert L.dpred_flush_bucket(4, 0, None, 0, t.ctypes.data, 0, None, 0, 0, None, 1, 1, 0, None, None, 0, None) == 0
    # the same call again (served by the plan cache), and with the overlap promise
    assert L.dpred_flush_bucket(4, 0, None, 0, t.ctypes.data, 0, None, 0, 0, None, 1, 1, 0, None, None, 0, None) == 0
    assert L.dpred_flush_bucket(4, 0, None, 0, t.ctypes.data, 0, None, 0, 0, None, 1, 1, 3, None, None, 0, None) == 0
    # unknown flag bits are rejected
    assert L.dpred_flush_bucket(4, 0, None, 0, t.ctypes.data, 0, None, 0, 0, None, 1, 1, 4, None, None, 0, None) == -1
    assert L.dpred_flush_workspace_bytes(8, 64) == 0          # 512 destinations at most: inline
    assert L.dpred_flush_workspace_bytes(8, 100) == 100 * 32 + 8 * 100 * 8
    assert L.dpred_flush_workspace_bytes(2, 200) == 200 * 32 + 2 * 200 * 8


def test_prepared_call_paths_agree_without_a_gpu(L):
    # BucketFlush reaches dpred_flush_bucket through the CPython call module
    # where it is built (it is here: this Python has headers) or through
    # ctypes; both give the same probe counters and the same errors.
    import torch
    assert zc._fast_call_module() is not None
    grads = torch.zeros((4, 64), dtype=torch.bfloat16)  # never touched: no call below launches
    empty = np.zeros(0, dtype=zc.TASK_DTYPE)
    seen = []
    for fast in (True, False):
        bf = zc.BucketFlush(grads, empty, None, None, fast=fast)
        assert bf.fast is fast
        assert bf(stream=0) is None
        seen.append(bf(stream=0, probe=True, flush_index=5))
    assert seen[0] == seen[1] == zc.Probe(5, 0, 0, 0, 0, [0, 0, 0, 0])
    errs = []
    for fast in (True, False):
        bad = zc.BucketFlush(grads, _tasks([(0, 0, 10)]), [9], None, fast=fast)  # owner 9 is not a rank
        for probe in (False, True):
            with pytest.raises(zc.DpredError) as e:
                bad(stream=0, probe=probe)
            errs.append((e.value.code, str(e.value)))
        # checked mode with a destination table: the table reaches the library
        # (a buffer on a non-owner rank is refused before any launch)
        tbl = zc.DstTable(4, 1, [0x20000, 0x30000, 0, 0])
        mis = zc.BucketFlush(grads, _tasks([(0, 0, 10)]), [0], tbl, checked=True, fast=fast)
        with pytest.raises(zc.DpredError) as e:
            mis(stream=0)
        assert e.value.code == -4 and "owned by rank 0" in str(e.value)
    assert len(set(errs)) == 1 and errs[0][0] == -1
    # zc.flush_bucket takes the module's one-shot call; forced onto ctypes it
    # gives the same probe and the same errors
    got = []
    for fast in (True, False):
        with pytest.MonkeyPatch.context() as mp:
            if not fast:
                mp.setattr(zc, "_FC", None)
                mp.setattr(zc, "_fast_call_module", lambda: None)
            got.append(zc.flush_bucket(grads, empty, None, None, probe=True, flush_index=7, stream=0))
            assert zc.flush_bucket(grads, empty, None, None, stream=0) is None
            with pytest.raises(zc.DpredError) as e:
                zc.flush_bucket(grads, _tasks([(0, 0, 10)]), [9], None, stream=0)
            got.append((e.value.code, str(e.value)))
            tbl = zc.DstTable(4, 1, [0x20000, 0x30000, 0, 0])
            with pytest.raises(zc.DpredError) as e:
                zc.flush_bucket(grads, _tasks([(0, 0, 10)]), [0], tbl, checked=True, probe=True, stream=0)
            got.append((e.value.code, str(e.value)))
    assert got[:3] == got[3:]
    assert got[0] == zc.Probe(7, 0, 0, 0, 0, [0, 0, 0, 0]) and got[1][0] == -1 and got[2][0] == -4
    fc = zc._fast_call_module()
    with pytest.raises(ValueError):
        fc.flush(object(), 0)                 # not a prepared call
    with pytest.raises(ValueError):
        fc.prepare(0, *([0] * 15))            # no function address
    with pytest.raises(TypeError):
        fc.flush(bf._cap)                     # stream missing
    with pytest.raises(TypeError):
        fc.call(0, 4)                         # 18 arguments
    with pytest.raises(ValueError):
        fc.call(*([0] * 17), None)            # no function address


def test_prepared_calls_from_several_threads_keep_their_own_errors(L):
    # the CPython module releases the interpreter lock during the call; the
    # library's error text is per thread, so concurrent failing calls each
    # read their own message
    import threading
    import torch
    grads = torch.zeros((4, 64), dtype=torch.bfloat16)  # never touched: every call fails validation
    bad = {k: zc.BucketFlush(grads, _tasks([(0, 0, 10)]), [o], None) for k, o in enumerate((4, 5, 6, 7))}
    seen, errors = {}, []

    def worker(k):
        try:
            for _ in range(500):
                with pytest.raises(zc.DpredError) as e:
                    bad[k](stream=0)
                seen.setdefault(k, set()).add(str(e.value))
        except Exception as exc:  # surfaced below
            errors.append(exc)
    threads = [threading.Thread(target=worker, args=(k,)) for k in bad]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors
    for k, msgs in seen.items():
        assert len(msgs) == 1, msgs
        assert str(4 + k) in next(iter(msgs))


def test_owner_map_argument_errors(L):
    own = np.zeros(2, np.int32)
    g = (zc._Group * 1)()
    n = np.array([5, 5], np.int64)
    g[0].comm_size, g[0].n_params, g[0].comm_ranks, g[0].numel = 2, 2, None, n.ctypes.data
    a, b = ctypes.c_int32(), ctypes.c_int32()
    assert L.dpred_build_owner_map(2, 2, g, 1, 1, own.ctypes.data, own.ctypes.data, own.ctypes.data,
                                   ctypes.byref(a), ctypes.byref(b)) == -1   # rank outside the world
    assert L.dpred_build_owner_map(0, 0, g, 1, 1, own.ctypes.data, own.ctypes.data, own.ctypes.data,
                                   ctypes.byref(a), ctypes.byref(b)) == -1
    n[1] = -3
    assert L.dpred_build_owner_map(2, 0, g, 1, 1, own.ctypes.data, own.ctypes.data, own.ctypes.data,
                                   ctypes.byref(a), ctypes.byref(b)) == -1


def test_partitioned_and_relayout_validation(L):
    tasks = _tasks([(0, 0, 10), (1, 10, 10)])
    flat = np.array([0, 10], np.int64)
    tbl = (ctypes.c_void_p * 2)(0x20000, 0x30000)
    used = np.zeros(2, np.int64)
    # a flat range beyond the world's partitions
    assert L.dpred_flush_bucket_partitioned(2, 0, 0x10000, 100, tasks.ctypes.data, 2, flat.ctypes.data, 2, 5, 0, tbl,
                                            1, None, None, 0, None) == -3
    # param id outside the offset table
    assert L.dpred_flush_bucket_partitioned(2, 0, 0x10000, 100, tasks.ctypes.data, 2, flat.ctypes.data, 1, 10, 0, tbl,
                                            1, None, None, 0, None) == -1
    # overlapping flat ranges
    bad = np.array([0, 5], np.int64)
    assert L.dpred_flush_bucket_partitioned(2, 0, 0x10000, 100, tasks.ctypes.data, 2, bad.ctypes.data, 2, 10, 0, tbl,
                                            1, None, None, 0, None) == -3
    # relayout: seg too small for a rank's run
    assert L.dpred_bucket_relayout(2, 0, 0x10000, 100, tasks.ctypes.data, 2, flat.ctypes.data, 2, 10, 5, 0x40000, 10,
                                   used.ctypes.data, None, 0, None) == -3
    # relayout: a partition's elements that are not one flat run
    gap = np.array([0, 12], np.int64)
    assert L.dpred_bucket_relayout(2, 0, 0x10000, 100, tasks.ctypes.data, 2, gap.ctypes.data, 2, 30, 30, 0x40000, 60,
                                   used.ctypes.data, None, 0, None) == -1


def test_executor_create_validates_and_destroys_without_a_gpu(L):
    """Creating an executor only builds host plans: no device call happens."""
    world = 4
    tasks = _tasks([(0, 0, 64), (1, 64, 64)])
    owner = np.array([0, -1], np.int32)
    starts = np.array([0], np.int64)
    counts = np.array([2], np.int32)
    dst = (ctypes.c_void_p * (world * 2))(*[0x100000 + 4096 * i for i in range(world * 2)])
    h = ctypes.c_void_p()
    # owner task with buffers on non-owner ranks is fine unchecked; a bad owner value is not
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 2, 0x10000, 128, 1, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, dst, None, 0, ctypes.byref(h)) == 0
    assert h.value
    assert L.dpred_executor_destroy(h) == 0
    bad_owner = np.array([7, -1], np.int32)
    assert L.dpred_executor_create(world, 0, 0, 1, 1, bad_owner.ctypes.data, 2, 0x10000, 128, 1, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, dst, None, 0, ctypes.byref(h)) == -1
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 2, 0x10000, 100, 1, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, dst, None, 0, ctypes.byref(h)) == -3
    # no destination table: in place, which needs the output dtype to be the input dtype
    assert L.dpred_executor_create(world, 0, 1, 1, 1, owner.ctypes.data, 2, 0x10000, 128, 1, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, None, None, 0, ctypes.byref(h)) == -1
    assert L.dpred_executor_flush(None, 0, None, None) == -1


def test_in_place_executor_without_a_gpu(L):
    """dst == NULL: results go back into the gradient rows.  Host plans only:
    validation, overlap eligibility and the refusal of host-buffer steps."""
    world, grads, ld = 4, 0x10000, 256
    owner = np.array([0, -1, 2], np.int32)
    tasks = _tasks([(0, 0, 64), (1, 64, 32), (2, 0, 100)])
    starts = np.array([0, 96], np.int64)
    counts = np.array([2, 1], np.int32)
    h = ctypes.c_void_p()
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 3, grads, ld, 2, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, None, None, 0, ctypes.byref(h)) == 0
    assert L.dpred_executor_overlap_eligible(h) == 1     # in-place writes stay in each bucket's own columns
    reg_dev = (ctypes.c_void_p * 1)(grads)
    reg_host = (ctypes.c_void_p * 1)(0x300000)
    nbytes = np.array([world * ld * 2], np.int64)
    assert L.dpred_executor_flush_all_from_host(h, 0x400000, ld, 1, reg_dev, reg_host, nbytes.ctypes.data, None,
                                                None) == -1
    assert L.dpred_executor_flush_all_mapped(h, 0x400000, ld, 1, reg_dev, reg_host, nbytes.ctypes.data, None,
                                             None) == -1
    assert "in-place" in L.dpred_last_error().decode()
    assert L.dpred_executor_destroy(h) == 0
    # two tasks of one bucket sharing columns cannot both be written in place
    overlapping = _tasks([(0, 0, 64), (1, 32, 32), (2, 0, 100)])
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 3, grads, ld, 2, starts.ctypes.data,
                                   counts.ctypes.data, overlapping.ctypes.data, None, None, 0, ctypes.byref(h)) == -3
    # bucket columns overlapping: allowed, but never overlapped on the GPU
    starts2 = np.array([0, 64], np.int64)
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 3, grads, ld, 2, starts2.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, None, None, 0, ctypes.byref(h)) == 0
    assert L.dpred_executor_overlap_eligible(h) == 0
    assert L.dpred_executor_destroy(h) == 0


def test_flush_path_and_pipeline_argument_errors(L):
    with pytest.raises(zc.DpredError):
        zc.set_flush_path(7)
    with pytest.raises(zc.DpredError):
        zc.set_allgather_form(7)
    prev = zc.set_allgather_form(zc.AG_STAGED)
    assert zc.set_allgather_form(prev) == zc.AG_STAGED
    # the write-only fill rejects bad arguments before any launch
    assert L.dpred_fill_pattern(0x200000, 64, 0, 3, 0, None) == -1             # unknown method
    assert L.dpred_fill_pattern(None, 64, 0, 0, 0, None) == -1                 # null destination
    assert L.dpred_fill_pattern(0x200008, 64, 0, 0, 0, None) == -2             # not 16-byte aligned
    assert L.dpred_fill_pattern(0x200010, 64, 0, 1, 0, None) == -2             # not 32-byte aligned
    assert L.dpred_fill_pattern(0x200000, 48, 0, 1, 0, None) == -2             # size not a multiple of 32
    assert L.dpred_fill_pattern(0x200000, 64, 0, 0, 33, None) == -1            # too many CTAs per SM
    assert L.dpred_fill_pattern(None, 0, 0, 0, 0, None) == 0                   # nothing to write
    assert L.dpred_stream_mixed(None, 0, None, 0, None) == 0                   # nothing to move
    assert L.dpred_stream_mixed(None, 16, 0x200000, 16, None) == -1            # null source
    assert L.dpred_stream_mixed(0x200000, 16, 0x300008, 16, None) == -2        # unaligned destination
    assert L.dpred_stream_mixed(0x200000, 24, 0x300000, 16, None) == -2        # size not a multiple of 16
    prev = zc.set_flush_path(zc.PATH_LDG)
    assert zc.set_flush_path(prev) == zc.PATH_LDG
    # the host pipeline rejects bad arguments before touching any stream
    world = 2
    tasks = _tasks([(0, 0, 32)])
    owner = np.array([0], np.int32)
    starts = np.array([0], np.int64)
    counts = np.array([1], np.int32)
    dst = (ctypes.c_void_p * 2)(0x200000, None)
    h = ctypes.c_void_p()
    assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 1, 0x10000, 64, 1, starts.ctypes.data,
                                   counts.ctypes.data, tasks.ctypes.data, dst, None, 0, ctypes.byref(h)) == 0
    reg_dev = (ctypes.c_void_p * 1)(0x200000)
    reg_host = (ctypes.c_void_p * 1)(0x300000)
    nbytes = np.array([64], np.int64)
    assert L.dpred_executor_flush_all_from_host(h, None, 64, 1, reg_dev, reg_host, nbytes.ctypes.data, None,
                                                None) == -1                     # no host gradients
    small = np.array([16], np.int64)                                            # destination outside every region
    assert L.dpred_executor_flush_all_from_host(h, 0x400000, 64, 1, reg_dev, reg_host, small.ctypes.data, None,
                                                None) == -1
    assert L.dpred_executor_flush(h, 3, None, None) == -1                      # bucket out of range
    assert L.dpred_executor_destroy(h) == 0


def test_executor_overlap_eligibility(L):
    """Consecutive flushes may overlap only when no two buckets can touch the
    same byte: disjoint columns, disjoint destinations, no destination inside
    the gradient array.  Host-only check at creation."""
    world, grads, ld = 2, 0x10000, 256          # gradient array [0x10000, 0x10400) in bf16
    owner = np.array([0, 1], np.int32)
    tasks = _tasks([(0, 0, 64), (1, 0, 64)])
    counts = np.array([1, 1], np.int32)

    def eligible(start1, dst_b1):
        starts = np.array([0, start1], np.int64)
        dst = (ctypes.c_void_p * 4)(0x100000, None, None, dst_b1)   # bucket 0: rank 0; bucket 1: rank 1
        h = ctypes.c_void_p()
        assert L.dpred_executor_create(world, 0, 0, 1, 1, owner.ctypes.data, 2, grads, ld, 2, starts.ctypes.data,
                                       counts.ctypes.data, tasks.ctypes.data, dst, None, 0, ctypes.byref(h)) == 0
        e = L.dpred_executor_overlap_eligible(h)
        if e == 1:
            assert L.dpred_executor_set_overlap(h, 0) == 1             # on by default
            assert L.dpred_executor_set_overlap(h, 1) == 0
        assert L.dpred_executor_destroy(h) == 0
        return e

    assert eligible(64, 0x200000) == 1
    assert eligible(32, 0x200000) == 0              # bucket columns [0, 64) and [32, 96) overlap
    assert eligible(64, grads + 512) == 0           # inside the gradient array, outside bucket 1's columns
    assert eligible(64, grads + 512 + 128) == 1     # inside the gradient array, in bucket 1's own columns (in place)
    assert eligible(64, grads + 512 + 130) == 0     # ... but running past them
    assert eligible(64, 0x100000 + 64) == 0         # bucket 1 writes into bucket 0's destination
    assert eligible(64, 0x100000 + 128) == 1        # adjacent, not overlapping
    assert L.dpred_executor_overlap_eligible(None) == -1
    assert L.dpred_executor_set_overlap(None, 1) == -1


def test_partitioned_executor_create_without_a_gpu(L):
    """The partitioned executor builds its plans on the host: valid buckets
    give an executor (eligible for launch overlap), and the partitioned
    flush's argument errors come back unchanged."""
    world, grads, ld = 2, 0x10000, 256
    tasks = _tasks([(0, 0, 64), (1, 64, 64)])          # params 0, 1 in one bucket; flat offsets 0, 64
    flat = np.array([0, 64], np.int64)
    starts = np.array([0], np.int64)
    counts = np.array([2], np.int32)
    parts = (ctypes.c_void_p * 2)(0x100000, 0x200000)
    h = ctypes.c_void_p()
    assert L.dpred_executor_create_partitioned(world, 0, 0, 1, grads, ld, 1, starts.ctypes.data, counts.ctypes.data,
                                               tasks.ctypes.data, flat.ctypes.data, 2, 64, parts, None, 0,
                                               ctypes.byref(h)) == 0
    assert L.dpred_executor_overlap_eligible(h) == 1
    assert L.dpred_executor_destroy(h) == 0
    assert L.dpred_executor_create_partitioned(world, 0, 0, 1, grads, ld, 1, starts.ctypes.data, counts.ctypes.data,
                                               tasks.ctypes.data, flat.ctypes.data, 2, 32, parts, None, 0,
                                               ctypes.byref(h)) == -3   # 128 elements do not fit 2 x 32
    assert L.dpred_executor_create_partitioned(world, 0, 0, 1, grads, ld, 1, starts.ctypes.data, counts.ctypes.data,
                                               tasks.ctypes.data, flat.ctypes.data, 2, 64, None, None, 0,
                                               ctypes.byref(h)) == -1   # no partition table
    assert L.dpred_executor_create_partitioned(world, 0, 0, 1, grads, 100, 1, starts.ctypes.data, counts.ctypes.data,
                                               tasks.ctypes.data, flat.ctypes.data, 2, 64, parts, None, 0,
                                               ctypes.byref(h)) == -3   # bucket wider than the row
