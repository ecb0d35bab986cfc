"""The native executor: its flushes equal single dpred_flush_bucket calls bit
for bit, the probe lines count flushes, and the host-buffer step (pipelined
host-to-device copies, flushes, device-to-host copies) returns exactly what
the device path computes."""
import warnings

import numpy as np
import pytest
import torch

import datagen
import zero_collectives_gb300 as zc
from datagen import BF16, F32, NORMAL, workloads
from tests.gpu_util import TORCH_DT, device_matrix, to_bits

pytestmark = pytest.mark.gpu


def _setup(world, tree, capacity, dt=torch.bfloat16, seed=5):
    layout = workloads.arrival_layout(tree, capacity=capacity)
    code = BF16 if dt == torch.bfloat16 else F32
    grads = device_matrix(world, tree.total, code, NORMAL, seed, sigma=1e-2)
    ex = zc.Zero1Executor(world, tree.numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets], dt,
                          fill=float("nan"))
    return layout, grads, ex


@pytest.mark.parametrize("world", [4, 8])
def test_executor_equals_single_calls(world):
    tree = workloads.straddle_tree(world, 40000 * world + 77, world - 1, pieces=5)
    layout, grads, ex = _setup(world, tree, capacity=tree.total // 3)
    assert len(layout.buckets) >= 3
    lines = []
    ex.probe_log = zc.ProbeLog(rank=0, sink=lines.append)
    probes = ex.flush_all(grads, probe=True)
    ref = zc.GradBuffers(world, ex.omap, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    for i, b in enumerate(layout.buckets):
        p = zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, ex.omap.owner, ref.dst_table(b.tasks), BF16,
                            True, True, probe=True)
        q = probes[i]
        assert (p.tasks, p.reduced_elems, p.owner_elems, p.kept_elems) == \
            (q.tasks, q.reduced_elems, q.owner_elems, q.kept_elems)
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(ex.grad.buf[r].view(torch.int16), ref.buf[r].view(torch.int16))
    assert [int(l.split("#")[1].split()[0]) for l in lines] == list(range(len(layout.buckets)))
    ex.flush_all(grads)   # the counter keeps going
    ex.close()


@pytest.mark.parametrize("mode", ["from_host", "mapped"])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_host_buffer_step_matches_device_path(dt, mode):
    world = 8
    tree = workloads.straddle_tree(world, 300000 * world + 5, 5, pieces=4)
    code = BF16 if dt == torch.bfloat16 else F32
    layout, grads_dev, ex = _setup(world, tree, capacity=tree.total // 4, dt=dt)
    ex.flush_all(grads_dev)
    torch.cuda.synchronize()
    want = [b.clone() for b in ex.grad.buf]
    host = torch.empty((world, tree.total), dtype=dt, pin_memory=True)
    arr = host.view(torch.int16 if dt == torch.bfloat16 else torch.int32).numpy()
    datagen.fill_host(arr.view(np.uint16 if dt == torch.bfloat16 else np.float32), code, NORMAL, 5, sigma=1e-2)
    outs = [torch.empty(b.shape, dtype=dt, pin_memory=True) for b in ex.grad.buf]
    scratch = torch.zeros_like(grads_dev)
    ex2 = zc.Zero1Executor(world, tree.numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets], dt,
                           fill=float("nan"))
    for _ in range(2):   # twice in a row: the pipeline's streams, or the mapped plans, are reused
        for o in outs:
            o.fill_(float("nan"))
        if mode == "from_host":
            ex2.flush_all_from_host(host, outs, scratch)
        else:
            ex2.flush_all_mapped(host, outs, scratch)
        torch.cuda.synchronize()
        if mode == "mapped":
            # nothing was staged: the device gradients and buffers were not touched
            assert not scratch.any()
            assert all(torch.isnan(b.float()).all() for b in ex2.grad.buf)
        for r in range(world):
            # everything a bucket wrote came back; the rest of the host buffer is untouched (NaN)
            w = want[r].cpu()
            written = ~torch.isnan(w.float())
            assert torch.equal(outs[r][written].view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                               w[written].view(torch.int16 if dt == torch.bfloat16 else torch.int32))
    ex.close()
    ex2.close()


def test_step_captured_in_a_cuda_graph():
    """A step whose plans travel inside the launches can be captured once and
    replayed: replays give the eager result bit for bit, and follow new data
    written into the same gradient tensor."""
    world = 8
    tree = workloads.straddle_tree(world, 20000 * world + 3, 4, pieces=3)
    layout, grads, ex = _setup(world, tree, capacity=tree.total // 2)
    ex.flush_all(grads)                      # eager: also does the one-time launch set-up
    torch.cuda.synchronize()
    eager = [b.clone() for b in ex.grad.buf]
    for b in ex.grad.buf:
        b.fill_(float("nan"))
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        ex.flush_all(grads)
    graph.replay()
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(ex.grad.buf[r].view(torch.int16), eager[r].view(torch.int16))
    # new gradients in the same tensor: the replay reduces them
    datagen.fill_device(grads.data_ptr(), world, tree.total, tree.total, BF16, NORMAL, 99, 0, 1, 0, 1e-2,
                        torch.cuda.current_stream().cuda_stream)
    graph.replay()
    fresh = zc.GradBuffers(world, ex.omap, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    for b in layout.buckets:
        zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, ex.omap.owner, fresh.dst_table(b.tasks), BF16,
                        True, True)
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(ex.grad.buf[r].view(torch.int16), fresh.buf[r].view(torch.int16))
    ex.close()


def test_work_runs_on_the_callers_stream():
    """Every entry point enqueues on the stream it is given: a flush on a side
    stream that waits on an event sees gradients written just before that
    event on another stream, and the default stream sees the flush's results
    only after waiting on the side stream."""
    world = 8
    tree = workloads.straddle_tree(world, 30000 * world + 1, 3, pieces=3)
    layout, grads, ex = _setup(world, tree, capacity=None)
    ref = zc.GradBuffers(world, ex.omap, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    b = layout.buckets[0]
    zc.flush_bucket(grads, b.tasks, ex.omap.owner, ref.dst_table(b.tasks), BF16, True, True)
    torch.cuda.synchronize()
    for buf in ex.grad.buf:
        buf.fill_(float("nan"))
    side = torch.cuda.Stream()
    ready = torch.cuda.Event()
    saved = grads.clone()
    grads.zero_()                                   # default stream
    grads.copy_(saved)
    ready.record(torch.cuda.current_stream())
    side.wait_event(ready)
    ex.flush_all(grads, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for r in range(world):
        assert torch.equal(ex.grad.buf[r].view(torch.int16), ref.buf[r].view(torch.int16))
    ex.close()


def test_mapped_step_rejects_pageable_host_memory():
    world = 4
    tree = workloads.straddle_tree(world, 5000 * world + 1, 2, pieces=2)
    layout, grads, ex = _setup(world, tree, capacity=tree.total // 2)
    pinned = torch.zeros((world, tree.total), dtype=torch.bfloat16, pin_memory=True)
    pageable = torch.zeros((world, tree.total), dtype=torch.bfloat16)
    outs = [torch.empty(b.shape, dtype=b.dtype, pin_memory=True) for b in ex.grad.buf]
    with pytest.raises(zc.DpredError) as e:
        ex.flush_all_mapped(pageable, outs, grads)
    assert e.value.code == -1                     # DPRED_E_INVAL
    with pytest.raises(zc.DpredError) as e:
        ex.flush_all_mapped(pinned, [torch.empty(b.shape, dtype=b.dtype) for b in ex.grad.buf], grads)
    assert e.value.code == -1
    short = torch.zeros((world, tree.total // 2), dtype=torch.bfloat16, pin_memory=True)
    with pytest.raises(zc.DpredError) as e:       # rows shorter than the buckets span
        ex.flush_all_mapped(short, outs, grads)
    assert e.value.code == -3                     # DPRED_E_SIZE
    assert zc.host_mapped_pointer(pinned) != 0
    ex.close()


@pytest.mark.parametrize("world", [2, 8, 16, 24, 64])  # persistent grids and one CTA per unit
def test_overlapped_launches_equal_serial_and_keep_stream_order(world):
    """Consecutive bucket flushes launched with programmatic stream
    serialisation give the serial result bit for bit, and work queued on the
    stream right after the step (a copy of every buffer) sees every bucket."""
    tree = workloads.straddle_tree(world, 150000 * world + 13, world - 1, pieces=6)
    layout, grads, ex = _setup(world, tree, capacity=tree.total // 6)
    assert len(layout.buckets) >= 5
    ex._bind(grads)
    assert zc.lib().dpred_executor_overlap_eligible(ex._native) == 1
    ex.set_overlap(False)
    ex.flush_all(grads)
    torch.cuda.synchronize()
    serial = [b.clone() for b in ex.grad.buf]
    ex.set_overlap(True)
    for _ in range(3):
        for b in ex.grad.buf:
            b.fill_(float("nan"))
        ex.flush_all(grads)
        after = [b.clone() for b in ex.grad.buf]   # same stream, queued right behind the last flush
        torch.cuda.synchronize()
        for r in range(world):
            assert torch.equal(after[r].view(torch.int16), serial[r].view(torch.int16))
    assert zc.device_status() == 0
    ex.close()


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("rto", [True, False])
@pytest.mark.parametrize("world,dt", [(8, torch.bfloat16), (4, torch.float32), (3, torch.bfloat16)])
def test_in_place_executor_matches_the_oracle(world, dt, rto, overlap):
    """The in-place executor step (no destination tables): every bucket's
    delivered results land in the gradient rows themselves, bit for bit as the
    oracle's in-place flush computes them, with W-1 straddlers and an
    excluded group; the probes count what each row received."""
    import oracle
    code = BF16 if dt == torch.bfloat16 else F32
    tree = workloads.straddle_tree(world, 30000 * world + 77, world - 1, pieces=4)
    ex_sizes = np.array([96, 64, 40], np.int64)
    numel = np.concatenate([tree.numel, ex_sizes])
    full = workloads.Tree([f"p{i}" for i in range(len(numel))], numel)
    layout = workloads.arrival_layout(full, capacity=full.total // 3)
    assert len(layout.buckets) >= 3
    sub = list(range(max(1, world // 2)))
    groups = [(None, tree.numel), (sub, ex_sizes)]
    grads = device_matrix(world, full.total, code, NORMAL, 13, sigma=1e-2)
    host = datagen.host_matrix(world, full.total, code, NORMAL, 13, sigma=1e-2)
    ex = zc.InPlaceExecutor(world, numel, [(b.start, b.tasks) for b in layout.buckets], dt, reduce_to_owner=rto,
                            groups=groups)
    ex.set_overlap(overlap)
    probes = ex.flush_all(grads, probe=True)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel), (sub, ex_sizes)], rto)
    assert np.array_equal(om["owner"], ex.omap.owner)
    for i, b in enumerate(layout.buckets):
        part = np.ascontiguousarray(host[:, b.start:b.start + b.size])
        op = oracle.flush(world, part, b.tasks, om["owner"], full.n_params, None, code, True, rto)
        host[:, b.start:b.start + b.size] = part
        q = probes[i]
        assert (q.tasks, q.reduced_elems, q.owner_elems, q.kept_elems) == \
            (op["tasks"], op["reduced_elems"], op["owner_elems"], op["kept_elems"])
    torch.cuda.synchronize()
    got = to_bits(grads)
    assert np.array_equal(got, host.view(np.uint16 if code == BF16 else np.uint32))
    assert zc.device_status() == 0
    assert ex._native is not None and zc.lib().dpred_executor_overlap_eligible(ex._native) == 1
    with pytest.raises(zc.DpredError):
        ex.flush_all_mapped(torch.empty(grads.shape, dtype=dt, pin_memory=True),
                            [torch.empty(1, dtype=dt, pin_memory=True) for _ in range(world)], grads)
    ex.close()


def test_per_call_capture_replays_and_uploaded_plans_are_refused():
    """Per-call flushes whose plans travel inside the launches can be captured
    with the overlap promise and replayed bit for bit.  A flush whose plan
    needs the workspace uploads it from host memory, which a graph cannot
    capture: under capture the call is refused before anything is enqueued,
    and the same call made eagerly works."""
    world = 8
    tree = workloads.straddle_tree(world, 20000 * world + 3, 4, pieces=3)
    layout = workloads.arrival_layout(tree, capacity=tree.total // 3)
    grads = device_matrix(world, tree.total, BF16, NORMAL, 5, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, tree.numel)], True)
    bufs = zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    tables = [bufs.dst_table(b.tasks) for b in layout.buckets]
    assert len(layout.buckets) >= 2
    assert all(zc.flush_workspace_bytes(world, len(b.tasks)) == 0 for b in layout.buckets)

    def step():
        for b, tab in zip(layout.buckets, tables):
            zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, om.owner, tab, BF16, True, True,
                            overlap=True)

    step()
    torch.cuda.synchronize()
    eager = [b.clone() for b in bufs.buf]
    for b in bufs.buf:
        b.fill_(float("nan"))
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    graph.replay()
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(bufs.buf[r].view(torch.int16), eager[r].view(torch.int16))

    # a 300-task bucket: its plan goes to the workspace
    sizes = np.array([(i * 53) % 700 + 1 for i in range(300)], np.int64)
    big = workloads.Tree([f"p{i}" for i in range(len(sizes))], sizes)
    b = workloads.arrival_layout(big, capacity=None).buckets[0]
    assert zc.flush_workspace_bytes(world, len(b.tasks)) > 0
    g2 = device_matrix(world, big.total, BF16, NORMAL, 6, sigma=1e-2)
    om2 = zc.build_owner_map(world, [(None, big.numel)], True)
    bufs2 = zc.GradBuffers(world, om2, big.numel, workloads.arrival_layout(big, capacity=None).row_offset,
                           torch.bfloat16, fill=float("nan"))
    tab2 = bufs2.dst_table(b.tasks)
    ws = torch.empty(zc.flush_workspace_bytes(world, len(b.tasks)), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    refused = torch.cuda.CUDAGraph()
    with warnings.catch_warnings():  # the capture ends empty, as it should
        warnings.simplefilter("ignore")
        with torch.cuda.graph(refused, stream=side):
            with pytest.raises(zc.DpredError) as err:
                zc.flush_bucket(g2, b.tasks, om2.owner, tab2, BF16, workspace=ws)
    assert err.value.code == -1 and "graph" in str(err.value)
    torch.cuda.synchronize()
    assert all(bool(torch.isnan(x.float()).all()) for x in bufs2.buf), "the refused call wrote something"
    zc.flush_bucket(g2, b.tasks, om2.owner, tab2, BF16, workspace=ws)
    torch.cuda.synchronize()
    assert not all(bool(torch.isnan(x.float()).all()) for x in bufs2.buf)
    assert zc.device_status() == 0
