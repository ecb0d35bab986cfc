"""Pins of the oracle's owner map (DeepSpeed issue #8700, "Design points").

Each test checks the oracle against something other than itself: element-by-
element brute force, the invariants the issue states (identical on every rank,
one owner per non-straddler, at most ws-1 straddlers per group, excluded
communicators, the flag-off path), and the straddlers of the 402.8M tree found
by scanning partition boundaries.
"""
import itertools

import numpy as np
import pytest

import oracle
from datagen import workloads


def brute_force(world, sizes):
    """Assign every element of the flat space to partition e // ceil(T/W), then
    read off each parameter's set of partitions."""
    T = int(sum(sizes))
    P = -(-T // world) if T else 0
    owner, lo, hi = [], [], []
    pos = 0
    for n in sizes:
        parts = sorted({e // P for e in range(pos, pos + n)}) if n else []
        pos += n
        if not parts:
            owner.append(-1), lo.append(-1), hi.append(-1)
        else:
            owner.append(parts[0] if len(parts) == 1 else -1)
            lo.append(parts[0])
            hi.append(parts[-1])
    return owner, lo, hi


def om(world, sizes, reduce_to_owner=True, rank=0, ranks=None):
    ranks = list(range(world)) if ranks is None else ranks
    return oracle.owner_map(world, [(ranks, np.asarray(sizes, np.int64))], reduce_to_owner, rank)


def test_brute_force_exhaustive_small():
    for world in range(1, 5):
        for n_params in range(1, 4):
            for sizes in itertools.product(range(0, 6), repeat=n_params):
                got = om(world, sizes)
                owner, lo, hi = brute_force(world, sizes)
                assert list(got["owner"]) == owner, (world, sizes)
                assert list(got["holder_lo"]) == lo and list(got["holder_hi"]) == hi, (world, sizes)


def test_brute_force_random():
    rng = np.random.default_rng(7)
    for _ in range(3000):
        world = int(rng.integers(1, 6))
        sizes = [int(v) for v in rng.integers(0, 9, size=int(rng.integers(1, 7)))]
        got = om(world, sizes)
        owner, lo, hi = brute_force(world, sizes)
        assert list(got["owner"]) == owner and list(got["holder_lo"]) == lo and list(got["holder_hi"]) == hi


def test_identical_on_every_rank():
    rng = np.random.default_rng(8)
    for world in (2, 4, 8, 16):
        sizes = rng.integers(1, 5000, size=50)
        ref = om(world, sizes, rank=0)
        for rank in range(world):
            got = om(world, sizes, rank=rank)
            for k in ("owner", "holder_lo", "holder_hi"):
                assert np.array_equal(got[k], ref[k])


def test_one_owner_per_non_straddler_and_element_balance():
    rng = np.random.default_rng(9)
    for world in (2, 3, 4, 8, 16):
        sizes = rng.integers(1, 10000, size=80)
        got = om(world, sizes)
        own, lo, hi = got["owner"], got["holder_lo"], got["holder_hi"]
        single = lo == hi
        assert np.array_equal(own[single], lo[single])
        assert np.all(own[~single] == -1)
        owned = sizes[own >= 0].sum()
        straddling = sizes[own < 0].sum()
        assert owned + straddling == sizes.sum()
        assert got["n_owned"] == int(single.sum()) and got["n_total"] == len(sizes)


def test_at_most_ws_minus_one_straddlers_per_group():
    rng = np.random.default_rng(10)
    for _ in range(300):
        world = int(rng.integers(2, 17))
        groups = []
        for g in range(int(rng.integers(1, 4))):
            groups.append((list(range(world)), rng.integers(1, 3000, size=int(rng.integers(1, 60)))))
        got = oracle.owner_map(world, groups)
        pos = 0
        for _, sizes in groups:
            seg = got["owner"][pos:pos + len(sizes)]
            assert (seg < 0).sum() <= world - 1
            pos += len(sizes)


def test_402m_tree_straddlers():
    """Straddlers found independently: the parameter that strictly contains each
    interior partition boundary j * ceil(T/8)."""
    tree = workloads.tree_402m()
    world = 8
    got = om(world, tree.numel)
    T = tree.total
    P = -(-T // world)
    starts = np.concatenate([[0], np.cumsum(tree.numel)])
    expected = set()
    for j in range(1, world):
        b = j * P
        for p in range(tree.n_params):
            if starts[p] < b < starts[p + 1]:
                expected.add(p)
    assert set(np.nonzero(got["owner"] < 0)[0].tolist()) == expected
    names = sorted(tree.names[p] for p in expected)
    assert names == sorted(["embed", "l0.q", "l4.q", "l8.q", "l12.q", "l16.q", "l20.q"])
    assert got["n_owned"] == 243 - 7 and got["n_total"] == 243
    # every straddler of this tree spans exactly two partitions
    strad = got["owner"] < 0
    assert np.all(got["holder_hi"][strad] - got["holder_lo"][strad] == 1)


@pytest.mark.parametrize("ranks", [[0, 1, 2, 3], [1, 0, 2, 3, 4, 5, 6, 7], [0, 2, 4, 6]])
def test_excluded_communicator(ranks):
    world = 8
    dp = np.array([100, 200, 300, 400, 500], np.int64)
    moe = np.array([64, 64, 64], np.int64)
    alone = oracle.owner_map(world, [(list(range(world)), dp)])
    both = oracle.owner_map(world, [(list(range(world)), dp), (ranks, moe)])
    assert np.array_equal(both["owner"][:5], alone["owner"])
    assert np.all(both["owner"][5:] == -1)
    assert np.all(both["holder_lo"][5:] == 0) and np.all(both["holder_hi"][5:] == world - 1)
    assert both["n_total"] == 8 and both["n_owned"] == alone["n_owned"]


def test_flag_off_declares_no_owner():
    tree = workloads.tree_402m()
    got = om(8, tree.numel, reduce_to_owner=False)
    assert np.all(got["owner"] == -1) and got["n_owned"] == 0
    on = om(8, tree.numel, reduce_to_owner=True)
    assert np.array_equal(got["holder_lo"], on["holder_lo"]) and np.array_equal(got["holder_hi"], on["holder_hi"])


def test_zero_sized_parameter():
    got = om(2, [10, 0, 10])
    assert got["owner"][1] == -1 and got["holder_lo"][1] == -1 and got["holder_hi"][1] == -1
    assert list(got["owner"]) == [0, -1, 1]
