"""The AllGather schedules of the page "AllGather" executed step by step on
the GPU: after every step each node's buffer holds exactly the chunks the
oracle's simulation of that schedule says (the N=4 ring table, the N=8
recursive-doubling table, the bidirectional ring), slots not yet received are
untouched, and the final layouts equal dpred_allgather's."""
import numpy as np
import pytest
import torch

import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, UNIFORM
from tests.gpu_util import TORCH_DT, device_matrix, to_bits

pytestmark = pytest.mark.gpu


def expected_holdings(schedule, N):
    """[steps + 1][N][N] chunk id per slot (-1 = not held), from the oracle."""
    if schedule == zc.SCHED_RING:
        return oracle.ring_steps(N)["hold"]
    if schedule == zc.SCHED_BIDIR_RING:
        return oracle.bidir_ring_steps(N)["hold"]
    rd = oracle.rd_steps(N)
    have = [{i} for i in range(N)]
    out = [[[i if c == i else -1 for c in range(N)] for i in range(N)]]
    for j in range(len(rd["partner"])):
        have = [have[i] | have[int(rd["partner"][j, i])] for i in range(N)]
        out.append([[c if c in have[i] else -1 for c in range(N)] for i in range(N)])
    return np.array(out)


@pytest.mark.parametrize("schedule", [zc.SCHED_RING, zc.SCHED_BIDIR_RING, zc.SCHED_RECURSIVE_DOUBLING])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_schedule_step_by_step(schedule, N, dt):
    if schedule == zc.SCHED_RECURSIVE_DOUBLING and N & (N - 1):
        with pytest.raises(zc.DpredError):
            zc.allgather_schedule_steps(schedule, N)
        return
    hold = expected_holdings(schedule, N)
    steps = zc.allgather_schedule_steps(schedule, N)
    assert steps == len(hold) - 1
    for S in (1, 777, 4096):
        x = device_matrix(N, S, dt, UNIFORM, 9)
        xs = to_bits(x).reshape(N, S)
        bufs = torch.full((N, N * S), float("nan"), dtype=TORCH_DT[dt], device="cuda")
        nan_bits = to_bits(bufs[0, :1])[0]
        zc.allgather_schedule_init(schedule, x, bufs)
        for s in range(steps + 1):
            if s > 0:
                zc.allgather_schedule_step(schedule, bufs, s)
            torch.cuda.synchronize()
            b = to_bits(bufs).reshape(N, N, S)
            for i in range(N):
                for c in range(N):
                    want = hold[s][i][c]
                    if want < 0:
                        assert np.all(b[i, c] == nan_bits), (s, i, c)
                    else:
                        assert np.array_equal(b[i, c], xs[want]), (s, i, c)
        ref = torch.empty_like(bufs)
        zc.allgather(x, ref, 1 if schedule == zc.SCHED_RING else 0)
        torch.cuda.synchronize()
        assert torch.equal(ref.view(torch.int16), bufs.view(torch.int16))


def test_ring_n4_is_the_page_table(golden_dir):
    """The N=4 ring on the GPU reproduces the page's table row by row."""
    rows = []
    for line in open(f"{golden_dir}/ring_allgather_n4.txt"):
        if line.strip() and not line.startswith("#"):
            rows.append([c.strip().split(",") for c in line.split("|")[1:]])
    x = torch.arange(4, dtype=torch.float32, device="cuda").view(4, 1)
    bufs = torch.full((4, 4), -1.0, device="cuda")
    zc.allgather_schedule_init(zc.SCHED_RING, x, bufs)
    letters = "ABCD"
    for s, row in enumerate(rows):
        if s:
            zc.allgather_schedule_step(zc.SCHED_RING, bufs, s)
        got = bufs.cpu().numpy()
        for i in range(4):
            assert [letters[int(v)] for v in got[i] if v >= 0] == row[i]
