"""Randomised parity of the bucket flush against the oracle.

Every case draws a world size (1..16, plus 64), element types, a task list
with gaps between tasks and a padded row stride, an owner per parameter
(a rank or -1), a destination table where any buffer may be empty and any
non-empty buffer may sit at any element alignment, pre-division and the
reduce-to-owner flag, and a kernel family.  The GPU result must equal the
oracle's bit for bit; buffers that are not delivered, and the canaries around
every buffer, must stay untouched."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, NORMAL
from tests.gpu_util import TORCH_DT, np_bits, to_bits
from tests.helpers import is_sentinel

pytestmark = pytest.mark.gpu

GUARD = 8


def one_case(rng, case):
    world = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 64]))
    in_dt = int(rng.integers(0, 2))
    out_dt = int(rng.integers(0, 2))
    n_tasks = int(rng.integers(1, 30))
    n_params = n_tasks + int(rng.integers(0, 5))
    params = rng.permutation(n_params)[:n_tasks]
    sizes = rng.integers(0, 2500, size=n_tasks)
    tiny = rng.random(n_tasks) < 0.3            # tasks that are all head and tail
    sizes[tiny] = rng.integers(0, 40, size=int(tiny.sum()))
    gaps = rng.integers(0, 20, size=n_tasks)
    tasks = np.zeros(n_tasks, dtype=zc.TASK_DTYPE)
    pos = int(rng.integers(0, 9))
    for t in range(n_tasks):
        tasks[t] = (int(params[t]), 0, pos, int(sizes[t]))
        pos += int(sizes[t]) + int(gaps[t])
    ld = pos + int(rng.integers(0, 17))
    owner = rng.integers(-1, world, size=n_params).astype(np.int32)
    rto = bool(rng.integers(0, 2))
    pre_div = bool(rng.integers(0, 2))
    path = int(rng.choice([zc.PATH_LDG, zc.PATH_TMA]))

    host = datagen.host_matrix(world, ld, in_dt, NORMAL, 1000 + case, sigma=1e-2)
    grads = torch.from_numpy(host.view(np.int16 if in_dt == BF16 else np.int32)).cuda().view(TORCH_DT[in_dt])

    # destination table: each (rank, task) buffer present with probability 0.6
    present = rng.random((world, n_tasks)) < 0.6
    dev_bufs, host_dst, ptrs, offs = {}, [[None] * n_tasks for _ in range(world)], [], {}
    esize = 2 if out_dt == BF16 else 4
    for r in range(world):
        for t in range(n_tasks):
            n = int(sizes[t])
            if not present[r, t]:
                ptrs.append(0)
                continue
            shift = int(rng.integers(0, 9))
            buf = torch.full((n + 2 * GUARD + 8,), float("nan"), dtype=TORCH_DT[out_dt], device="cuda")
            dev_bufs[(r, t)] = buf
            offs[(r, t)] = GUARD + shift
            ptrs.append(buf.data_ptr() + (GUARD + shift) * esize)
            host_dst[r][t] = np.full(n, 0x7FC1, np.uint16) if out_dt == BF16 else \
                np.full(n, np.uint32(0x7FC00123), np.uint32).view(np.float32)
    table = zc.DstTable(world, n_tasks, ptrs)

    prev = zc.set_flush_path(path)
    try:
        ws = torch.empty(max(zc.flush_workspace_bytes(world, n_tasks), 16), dtype=torch.uint8, device="cuda")
        pr = zc.flush_bucket(grads, tasks, owner, table, out_dt, pre_div, rto, probe=True, workspace=ws)
    finally:
        zc.set_flush_path(prev)
    opr = oracle.flush(world, host.copy(), tasks, owner, n_params, host_dst, out_dt, pre_div, rto)
    torch.cuda.synchronize()
    for (r, t), buf in dev_bufs.items():
        n, s = int(sizes[t]), offs[(r, t)]
        got = to_bits(buf)
        isn = torch.isnan(buf.float()).cpu().numpy()
        assert isn[:s].all() and isn[s + n:].all(), f"case {case}: canary of rank {r} task {t}"
        want = host_dst[r][t]
        if n and np.all(is_sentinel(want, out_dt == BF16)):
            assert isn[s:s + n].all(), f"case {case}: rank {r} task {t} written but not delivered"
        else:
            assert np.array_equal(got[s:s + n], np_bits(want)), f"case {case}: rank {r} task {t} (W={world})"
    assert pr.kept_elems == opr["kept_elems"] and pr.owner_elems == opr["owner_elems"]


def test_flush_fuzz():
    rng = np.random.default_rng(2026)
    for case in range(300):
        one_case(rng, case)
    assert zc.device_status() == 0
