"""Pins of the oracle's partitioned (ReduceScatter-shaped) flush and of the
bucket relayout pass (DeepSpeed issue #8700, "Describe alternatives you've
considered": ncclReduceScatter over a bucket laid out by destination rank;
"Follow-up": ZeRO-2's real buffers with offsets).

Checked against: the element reduction applied to the bucket put in flat
order by numpy (concatenated partitions == reduced flat space); the owner
flush on the owner's buffer (same bits for parameters inside one partition);
ReduceScatter of the relayout (eq. ag-allreduce-decomposition's
ReduceScatter half); and the probe's element balance."""
import numpy as np
import pytest

import oracle
from datagen import BF16, F32, NORMAL, host_matrix, workloads
from tests.helpers import holder_sets, oracle_dst


def _case(world, elems, straddlers, in_dt=BF16, seed=3):
    tree = workloads.straddle_tree(world, elems, straddlers)
    layout = workloads.arrival_layout(tree, capacity=None)
    b = layout.buckets[0]
    grads = host_matrix(world, b.size, in_dt, NORMAL, seed, sigma=1e-2)
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    P = -(-tree.total // world)
    return tree, b, grads, flat, P


def _partitions(world, P, out_dt):
    return [np.full(P, 0x7FC1 if out_dt == BF16 else np.nan, dtype=np.uint16 if out_dt == BF16 else np.float32)
            for _ in range(world)]


@pytest.mark.parametrize("world,straddlers", [(2, 1), (4, 0), (4, 3), (8, 7), (5, 2)])
@pytest.mark.parametrize("out_dt", [BF16, F32])
def test_partitions_concatenate_to_the_reduced_flat_space(world, straddlers, out_dt):
    tree, b, grads, flat, P = _case(world, 3000 * world + 11, straddlers)
    parts = _partitions(world, P, out_dt)
    pr = oracle.flush_partitioned(world, grads, b.tasks, flat, P, parts, out_dt, pre_div=True)
    # the bucket in flat (model) order, built by numpy from the task table
    cols = np.empty(tree.total, np.int64)
    for t in b.tasks:
        s = flat[int(t["param_id"])]
        cols[s:s + int(t["numel"])] = np.arange(int(t["offset"]), int(t["offset"]) + int(t["numel"]))
    want = oracle.reduce_rows(np.ascontiguousarray(grads[:, cols]), pre_div=True, out_dt=out_dt)
    got = np.concatenate(parts)[:tree.total]
    assert np.array_equal(got.view(want.dtype), want)
    assert sum(pr["kept_elems"]) == pr["reduced_elems"] == tree.total
    strad = sum(int(t["numel"]) for t in b.tasks
                if flat[int(t["param_id"])] // P != (flat[int(t["param_id"])] + int(t["numel"]) - 1) // P)
    assert pr["owner_elems"] == tree.total - strad


def test_owner_parameters_match_the_owner_flush():
    world = 8
    tree, b, grads, flat, P = _case(world, 4000 * world + 5, 5)
    parts = _partitions(world, P, BF16)
    oracle.flush_partitioned(world, grads, b.tasks, flat, P, parts, BF16, True)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)], True)
    dst = oracle_dst(world, b.tasks, holder_sets(om["holder_lo"], om["holder_hi"]), True)
    oracle.flush(world, grads.copy(), b.tasks, om["owner"], tree.n_params, dst, BF16, True, True)
    for t, task in enumerate(b.tasks):
        p, n = int(task["param_id"]), int(task["numel"])
        r = om["owner"][p]
        if r >= 0:
            s = flat[p] - r * P
            assert np.array_equal(parts[r][s:s + n], dst[r][t])
        else:   # a straddler: each holder's partition gets its own slice of the full reduced parameter
            full = dst[om["holder_lo"][p]][t]
            for h in range(om["holder_lo"][p], om["holder_hi"][p] + 1):
                lo, hi = max(flat[p], h * P), min(flat[p] + n, (h + 1) * P)
                assert np.array_equal(parts[h][lo - h * P:hi - h * P], full[lo - flat[p]:hi - flat[p]])


@pytest.mark.parametrize("world,straddlers", [(2, 1), (4, 3), (8, 0), (8, 7)])
def test_relayout_then_reduce_scatter_is_the_partitioned_flush(world, straddlers):
    tree, b, grads, flat, P = _case(world, 2500 * world + 3, straddlers)
    seg = P
    out = np.zeros((world, world * seg), np.uint16)
    used = oracle.bucket_relayout(grads, b.tasks, flat, P, seg, out)
    assert int(used.sum()) == tree.total
    rs = oracle.reduce_scatter(out, pre_div=True)
    parts = _partitions(world, P, BF16)
    oracle.flush_partitioned(world, grads, b.tasks, flat, P, parts, BF16, True)
    for r in range(world):
        assert np.array_equal(rs[r][:used[r]], parts[r][:used[r]])
    # the relayout is a permutation of each replica row
    for q in range(world):
        moved = np.concatenate([out[q, r * seg:r * seg + used[r]] for r in range(world)])
        assert np.array_equal(np.sort(moved), np.sort(grads[q]))


def test_partitioned_flush_on_the_402m_bucket_tree():
    """Probe balance over the seven buckets of the 402.8M model at W=8: every
    element reaches exactly one rank."""
    tree = workloads.tree_402m()
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    P = -(-tree.total // 8)
    L = workloads.arrival_layout(tree)
    b = L.buckets[1]
    g = np.zeros((8, b.size), np.uint16)
    parts = [None] * 8   # counters only: no rank receives values
    pr = oracle.flush_partitioned(8, g, b.tasks, flat, P, parts, BF16, True)
    assert pr["reduced_elems"] == b.size and pr["owner_tasks"] == len(b.tasks) - 1
