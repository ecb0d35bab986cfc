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
