"""Pins of the oracle's ReduceScatter / AllGather and the schedules of the page
"AllGather" (tier6-model interconnect notes): the worked N=4 ring table and
N=8 recursive-doubling table, AllReduce = ReduceScatter + AllGather, per-node
receive (N-1)M/N, and the cost closed forms."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from datagen import BF16, F32, UNIFORM, host_matrix, workloads
from tests.helpers import bits


def _read_table(path):
    rows = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([c.strip() for c in line.split("|")])
    return rows


def test_ring_n4_matches_worked_table(golden_dir):
    rows = _read_table(f"{golden_dir}/ring_allgather_n4.txt")
    sim = oracle.ring_steps(4)
    letters = "ABCD"
    for s, row in enumerate(rows):
        for i in range(4):
            want = row[1 + i].split(",")
            got = [letters[c] for c in sim["hold"][s, i] if c >= 0]
            assert got == want, (row[0], i)
    final = [[letters[c] for c in sim["hold"][3, i]] for i in range(4)]
    # the ring-order AllGather layout equals the schedule's final holdings
    x = np.arange(4, dtype=np.float32).reshape(4, 1)
    ag = oracle.allgather(x, order=1)
    assert [[letters[int(v)] for v in ag[i]] for i in range(4)] == final


def test_rd_n8_matches_worked_table(golden_dir):
    rows = _read_table(f"{golden_dir}/rd_allgather_n8.txt")
    sim = oracle.rd_steps(8)
    N = 8
    for j, row in enumerate(rows):
        pairs = {tuple(sorted((i, int(sim["partner"][j, i])))) for i in range(N)}
        want = {tuple(int(v) for v in p.strip("()").split(",")) for p in row[1].replace(")(", ") (").split()}
        assert pairs == want
        assert Fraction(int(sim["xfer_chunks"][j]), N) == Fraction(row[2])
        assert Fraction(int(sim["held_chunks"][j]), N) == Fraction(row[3])
    assert np.array_equal(sim["final"], np.tile(np.arange(N), (N, 1)))


@pytest.mark.parametrize("N", [2, 3, 4, 5, 8, 16])
def test_per_node_receive(N):
    M = N * 65536
    ring = oracle.ring_steps(N)
    assert np.all(ring["recv_chunks"] * (M // N) == oracle.ag_recv(N, M))
    if N & (N - 1) == 0:
        rd = oracle.rd_steps(N)
        assert np.all(rd["recv_chunks"] * (M // N) == oracle.ag_recv(N, M))
        assert sum(2 ** (j - 1) for j in range(1, int(math.log2(N)) + 1)) == N - 1
        assert list(rd["xfer_chunks"]) == [2 ** (j - 1) for j in range(1, int(math.log2(N)) + 1)]
    else:
        with pytest.raises(ValueError):
            oracle.rd_steps(N)


def test_cost_closed_forms_at_n8():
    a, b, M = 1.0, 1.0, 8.0
    assert oracle.ring_ag_time(8, M, a, b) == 7 * a + 7 * M / (8 * b)
    assert oracle.bidir_ring_ag_time(8, M, a, b) == 4 * (a + M / (8 * b))
    assert oracle.rd_ag_time(8, M, a, b) == 3 * a + 7 * M / (8 * b)
    # recursive doubling meets both lower bounds; ring meets the bandwidth one
    assert oracle.rd_ag_time(8, M, a, b) == oracle.ag_latency_lower_bound(8, a) + oracle.ag_bw_lower_bound(8, M, 1, b)
    assert oracle.ring_ag_time(8, M, 0.0, b) == oracle.ag_bw_lower_bound(8, M, 1, b)
    assert oracle.ag_latency_lower_bound(5, 1.0) == 3


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_reduce_scatter_then_allgather_is_allreduce(N, dt):
    M = N * 3000
    x = host_matrix(N, M, dt, UNIFORM, seed=5)
    rs = oracle.reduce_scatter(x)
    ag = oracle.allgather(rs, order=0)
    ar = x.copy()
    tasks = np.zeros(1, dtype=workloads.TASK_DTYPE)
    tasks["numel"] = M
    oracle.flush(N, ar, tasks, None, 1, None, dt, pre_div=False, reduce_to_owner=False)
    for i in range(N):
        assert np.array_equal(bits(ag[i]), bits(ar[i]))


def test_reduce_scatter_is_shard_of_reduction():
    N, M = 4, 4 * 1001
    x = host_matrix(N, M, BF16, UNIFORM, seed=6)
    rs = oracle.reduce_scatter(x, pre_div=True)
    full = oracle.reduce_rows(x, pre_div=True)
    assert np.array_equal(rs.reshape(-1), full)
    with pytest.raises(ValueError):
        oracle.reduce_scatter(x[:, :M - 1])


@pytest.mark.parametrize("order", [0, 1])
def test_allgather_is_a_pure_copy(order):
    N, S = 8, 777
    rng = np.random.default_rng(3)
    x = rng.integers(0, 2**16, size=(N, S), dtype=np.uint64).astype(np.uint16)  # includes NaN patterns
    out = oracle.allgather(x, order)
    for i in range(N):
        for c in range(N):
            src = c if order == 0 else (i - c) % N
            assert np.array_equal(out[i, c * S:(c + 1) * S], x[src])


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 9, 16])
def test_bidirectional_ring_steps_and_receive(N):
    """eq. ag-bidir-ring: ceil((N-1)/2) steps; every node ends with all chunks
    and receives (N-1)/N of M (eq. allgather-recv)."""
    sim = oracle.bidir_ring_steps(N)
    assert sim["steps"] == math.ceil((N - 1) / 2)
    assert np.array_equal(sim["hold"][-1], np.tile(np.arange(N), (N, 1)))
    assert np.all(sim["recv_chunks"] == N - 1)
    # each step adds at most two chunks per node
    for s in range(1, sim["steps"] + 1):
        grown = (sim["hold"][s] >= 0).sum(axis=1) - (sim["hold"][s - 1] >= 0).sum(axis=1)
        assert np.all((grown >= 1) & (grown <= 2))


def test_bidirectional_ring_n4_by_hand():
    sim = oracle.bidir_ring_steps(4)
    held = lambda s, i: [int(c) for c in sim["hold"][s, i] if c >= 0]  # noqa: E731
    assert held(1, 0) == [0, 1, 3]          # A gets B from the right and D from the left
    assert held(2, 0) == [0, 1, 2, 3]       # C arrives from both sides at once
    assert held(1, 2) == [1, 2, 3]


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_product_cost_model_agrees_with_the_oracle_forms(N):
    from zero_collectives_gb300 import costs
    M, a, b = 1e9, 3e-6, 5e10
    assert costs.ring(N, M, a, b) == pytest.approx(oracle.ring_ag_time(N, M, a, b))
    assert costs.bidirectional_ring(N, M, a, b) == pytest.approx(oracle.bidir_ring_ag_time(N, M, a, b))
    assert costs.recursive_doubling(N, M, a, b) == pytest.approx(oracle.rd_ag_time(N, M, a, b))
    lat, bw = costs.lower_bounds(N, M, a, b)
    assert lat == pytest.approx(oracle.ag_latency_lower_bound(N, a)) and bw == pytest.approx(oracle.ag_bw_lower_bound(N, M, 1, b))
