"""GPU parity of the partitioned (ReduceScatter-shaped) flush and of the bucket
relayout pass against the oracle, relayout + ReduceScatter against the fused
flush, and the full 402.8M-parameter W=8 partitioned flush (every partition
element written exactly once, sampled values checked one by one)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, NORMAL, workloads
from tests.gpu_util import TORCH_DT, device_matrix, np_bits, to_bits

pytestmark = pytest.mark.gpu

GUARD = 16


@pytest.fixture(params=[zc.PATH_LDG, zc.PATH_TMA], ids=["ldg", "tma"], autouse=True)
def flush_path(request):
    prev = zc.set_flush_path(request.param)
    yield request.param
    zc.set_flush_path(prev)


def _case(world, elems, straddlers, capacity=None):
    tree = workloads.straddle_tree(world, elems, straddlers)
    layout = workloads.arrival_layout(tree, capacity=capacity)
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    P = -(-tree.total // world)
    return tree, layout, flat, P


@pytest.mark.parametrize("world", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("in_dt,out_dt", [(BF16, BF16), (F32, F32), (BF16, F32)])
def test_partitioned_flush_matches_oracle(world, in_dt, out_dt):
    for straddlers, shift in ((world - 1, 0), (world // 2, 1)):
        tree, layout, flat, P = _case(world, 5000 * world + 9, straddlers)
        b = layout.buckets[0]
        grads = device_matrix(world, tree.total, in_dt, NORMAL, 13, sigma=1e-2)
        host = datagen.host_matrix(world, tree.total, in_dt, NORMAL, 13, sigma=1e-2)
        bufs = [torch.full((P + 2 * GUARD,), float("nan"), dtype=TORCH_DT[out_dt], device="cuda")
                for _ in range(world)]
        views = [bb[GUARD + shift:GUARD + shift + P] for bb in bufs]
        ws = torch.empty(max(zc.flush_workspace_bytes(world, len(b.tasks) + world - 1), 16), dtype=torch.uint8,
                         device="cuda")
        pr = zc.flush_bucket_partitioned(grads, b.tasks, flat, P, views, out_dt, True, probe=True, workspace=ws)
        parts = [np.full(P, 0, dtype=np.uint16 if out_dt == BF16 else np.float32) for _ in range(world)]
        opr = oracle.flush_partitioned(world, host, b.tasks, flat, P, parts, out_dt, True)
        torch.cuda.synchronize()
        for r in range(world):
            got = to_bits(bufs[r])
            used = opr["kept_elems"][r]
            lo = GUARD + shift
            assert np.array_equal(got[lo:lo + used], np_bits(parts[r])[:used]), f"rank {r}"
            isn = torch.isnan(bufs[r].float()).cpu().numpy()
            assert isn[:lo].all() and isn[lo + used:].all(), f"rank {r}: write outside its slice"
        assert pr.kept_elems == opr["kept_elems"] and pr.owner_elems == opr["owner_elems"]


@pytest.mark.parametrize("world", [2, 4, 8])
def test_relayout_matches_oracle_and_feeds_reduce_scatter(world):
    tree, layout, flat, P = _case(world, 3000 * world + 17, world - 1)
    b = layout.buckets[0]
    rng = np.random.default_rng(world)
    host = rng.integers(0, 1 << 16, size=(world, tree.total), dtype=np.uint64).astype(np.uint16)  # any bits, NaNs too
    grads = torch.from_numpy(host.view(np.int16)).cuda().view(torch.bfloat16)
    seg = P
    out = torch.zeros((world, world * seg), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(zc.bucket_relayout_workspace_bytes(world, len(b.tasks)), 16), dtype=torch.uint8,
                     device="cuda")
    used = zc.bucket_relayout(grads, b.tasks, flat, P, seg, out, workspace=ws)
    want = np.zeros((world, world * seg), np.uint16)
    oused = oracle.bucket_relayout(host, b.tasks, flat, P, seg, want)
    torch.cuda.synchronize()
    assert np.array_equal(used, oused)
    assert np.array_equal(to_bits(out), want)
    # finite data for the reduction: relayout + ReduceScatter == fused partitioned flush
    g2 = device_matrix(world, tree.total, BF16, NORMAL, 21, sigma=1e-2)
    out.zero_()
    zc.bucket_relayout(g2, b.tasks, flat, P, seg, out, workspace=ws)
    rs = torch.empty((world, seg), dtype=torch.bfloat16, device="cuda")
    zc.reduce_scatter(out, rs, pre_div=True)
    parts = [torch.full((P,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    wsf = torch.empty(max(zc.flush_workspace_bytes(world, len(b.tasks) + world - 1), 16), dtype=torch.uint8,
                      device="cuda")
    zc.flush_bucket_partitioned(g2, b.tasks, flat, P, parts, BF16, True, workspace=wsf)
    torch.cuda.synchronize()
    for r in range(world):
        u = int(used[r])
        assert torch.equal(rs[r, :u].view(torch.int16), parts[r][:u].view(torch.int16))


def test_402m_w8_partitioned_full_size_sampled():
    world, seed, sigma = 8, 3, 1e-3
    tree = workloads.tree_402m()
    layout = workloads.arrival_layout(tree)
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    P = -(-tree.total // world)
    grads = device_matrix(world, tree.total, BF16, NORMAL, seed, sigma=sigma)
    parts = [torch.full((P,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    for b in layout.buckets:
        zc.flush_bucket_partitioned(grads[:, b.start:b.start + b.size], b.tasks, flat, P, parts, BF16, True)
    torch.cuda.synchronize()
    for r in range(world):
        n_r = min(P, tree.total - r * P)
        assert int(torch.isnan(parts[r][:n_r].float()).sum().item()) == 0, f"rank {r}: unwritten elements"
    rng = np.random.default_rng(5)
    f = np.unique(np.concatenate([[0, P - 1, P, tree.total - 1], rng.integers(0, tree.total, size=20000)]))
    # flat position -> column of the arrival-order row
    starts = flat
    pid = np.searchsorted(starts, f, side="right") - 1
    cols = layout.row_offset[pid] + (f - starts[pid])
    x = np.stack([datagen.sample_host(np.full(len(cols), r), cols, BF16, NORMAL, seed, sigma) for r in range(world)])
    want = oracle.reduce_rows(x, pre_div=True)
    rank = f // P
    for r in range(world):
        sel = rank == r
        idx = torch.from_numpy((f[sel] - r * P).astype(np.int64)).cuda()
        assert np.array_equal(to_bits(parts[r][idx]), want[sel]), f"rank {r}"


@pytest.mark.parametrize("world", [4, 8])
def test_partitioned_executor_matches_oracle_and_single_calls(world):
    """The partitioned executor over several arrival-order buckets: every
    partition equals the oracle's, bit for bit, with the launch overlap on and
    off and through the mapped host step; probes equal the single calls'."""
    tree = workloads.straddle_tree(world, 60000 * world + 31, world - 1, pieces=5)
    layout = workloads.arrival_layout(tree, capacity=tree.total // 5)
    assert len(layout.buckets) >= 4
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    grads = device_matrix(world, tree.total, BF16, NORMAL, 17, sigma=1e-2)
    host = datagen.host_matrix(world, tree.total, BF16, NORMAL, 17, sigma=1e-2)
    ex = zc.PartitionedExecutor(world, tree.numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets],
                                torch.bfloat16)
    P = ex.part_size
    want = [np.zeros(P, np.uint16) for _ in range(world)]
    for b in layout.buckets:
        oracle.flush_partitioned(world, host[:, b.start:b.start + b.size].copy(), b.tasks, flat, P, want, BF16, True)
    ex._bind(grads)
    assert zc.lib().dpred_executor_overlap_eligible(ex._native) == 1
    for overlap in (False, True):
        ex.set_overlap(overlap)
        for p in ex.parts:
            p.fill_(float("nan"))
        probes = ex.flush_all(grads, probe=True)
        torch.cuda.synchronize()
        for r in range(world):
            used = min(P, max(0, tree.total - r * P))     # the last partition is shorter
            got = to_bits(ex.parts[r])
            assert np.array_equal(got[:used], want[r][:used]), f"rank {r}, overlap {overlap}"
            assert torch.isnan(ex.parts[r][used:].float()).all()
    ws = torch.empty(zc.flush_workspace_bytes(world, max(len(b.tasks) for b in layout.buckets) + world), dtype=torch.uint8,
                     device="cuda")
    scratch = [torch.empty(P, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    for i, b in enumerate(layout.buckets):
        pr = zc.flush_bucket_partitioned(grads[:, b.start:b.start + b.size], b.tasks, flat, P, scratch, BF16, True,
                                         probe=True, workspace=ws)
        q = probes[i]
        assert (pr.tasks, pr.reduced_elems, pr.owner_elems, pr.kept_elems) == \
            (q.tasks, q.reduced_elems, q.owner_elems, q.kept_elems)
    # the mapped host step: gradients and partitions in pinned host memory
    hg = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).pin_memory()
    outs = [torch.full((P,), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(world)]
    ex.flush_all_mapped(hg, outs, grads)
    torch.cuda.synchronize()
    for r in range(world):
        used = min(P, max(0, tree.total - r * P))
        assert np.array_equal(outs[r].view(torch.int16).numpy().view(np.uint16)[:used], want[r][:used]), \
            f"mapped, rank {r}"
    assert zc.device_status() == 0
    ex.close()
