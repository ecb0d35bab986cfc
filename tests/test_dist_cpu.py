"""The multi-rank host path of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job value, and the reference arm does no
work on ranks other than 0."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    elapsed = [12.5, 20.0][rank]
    m = bench.max_over_ranks(elapsed, world, device="cpu")
    v = bench.job_gbs(world, 7_463_473_152, 10, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 20.0
    assert v == pytest.approx(2 * 7_463_473_152 * 10 / 0.020 / 1e9)


def test_reference_arm_is_silent_off_rank_zero(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, max_buckets = 1, 1, 0
    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def _map_rank(rank, world, port, perturb, out):
    import numpy as np
    import zero_collectives_gb300 as zc
    from zero_collectives_gb300 import dist as zdist
    from datagen import workloads
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    sizes = workloads.tree_402m().numel.copy()
    if perturb and rank == 1:
        sizes[1] += 3_000_000    # rank 1 read a different parameter size: partition boundaries move
    omap = zc.build_owner_map(8, [(None, sizes)])
    try:
        out[rank] = ("ok", hex(zdist.check_owner_map(omap)))
    except zc.DpredError as e:
        out[rank] = ("mismatch", e.code)
    dist.destroy_process_group()


@pytest.mark.parametrize("perturb", [False, True])
def test_owner_map_consistency_across_ranks(perturb):
    """Two gloo ranks: identical metadata agrees; a rank with a different
    parameter size is detected on both ranks before any flush."""
    from zero_collectives_gb300 import build
    build.build()
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_map_rank, args=(2, port, perturb, out), nprocs=2, join=True)
    if perturb:
        assert out[0] == ("mismatch", -4) and out[1] == ("mismatch", -4)
    else:
        assert out[0][0] == "ok" and out[0] == out[1]


def test_digest_changes_with_the_map():
    import numpy as np
    import zero_collectives_gb300 as zc
    from zero_collectives_gb300 import build
    build.build()
    a = zc.build_owner_map(8, [(None, np.array([100, 200, 300, 400], np.int64))])
    b = zc.build_owner_map(8, [(None, np.array([100, 200, 300, 400], np.int64))])
    c = zc.build_owner_map(8, [(None, np.array([100, 200, 300, 400], np.int64))], reduce_to_owner=False)
    assert a.digest() == b.digest() != c.digest()
