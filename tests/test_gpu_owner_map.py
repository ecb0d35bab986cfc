"""The device owner map against the oracle and the host map, bit for bit:
the 402.8M tree, random groups spanning several 1024-parameter chunks with
zero-size parameters, excluded communicators and the flag-off path."""
import numpy as np
import pytest
import torch

import oracle
import zero_collectives_gb300 as zc
from datagen import workloads

pytestmark = pytest.mark.gpu


def check(world, sizes, ranks=None, rto=True):
    sizes = np.asarray(sizes, np.int64)
    o, lo, hi, counts = zc.build_owner_map_device(
        world, torch.from_numpy(sizes).cuda(),
        None if ranks is None else torch.tensor(ranks, dtype=torch.int32, device="cuda"), rto)
    torch.cuda.synchronize()
    ref = oracle.owner_map(world, [(list(range(world)) if ranks is None else ranks, sizes)], rto)
    assert np.array_equal(o.cpu().numpy(), ref["owner"])
    assert np.array_equal(lo.cpu().numpy(), ref["holder_lo"]) and np.array_equal(hi.cpu().numpy(), ref["holder_hi"])
    assert counts.cpu().tolist() == [ref["n_owned"], ref["n_total"]]
    host = zc.build_owner_map(world, [(ranks, sizes)], rto)
    assert np.array_equal(host.owner, ref["owner"])


def test_402m_tree():
    tree = workloads.tree_402m()
    check(8, tree.numel)
    check(8, tree.numel, rto=False)


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16, 64])
def test_random_groups_over_several_chunks(world):
    rng = np.random.default_rng(world)
    for n in (1, 31, 1024, 1025, 5000):
        sizes = rng.integers(0, 3000, size=n)
        sizes[rng.random(n) < 0.05] = 0
        check(world, sizes)


def test_excluded_and_empty_groups():
    check(8, [100, 200, 300], ranks=[0, 1, 2, 3])
    check(4, [100, 200, 300], ranks=[1, 0, 2, 3])
    check(4, [0, 0, 0])
    check(4, [])
