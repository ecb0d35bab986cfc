"""The allocation-free flush entry point (dpred_flush_bucket_noalloc).

It exists for callers that cannot allocate device memory -- runtimes working
inside a fixed device budget, plug-ins living inside another framework's
allocator.  Instead of a caller
workspace it keeps large task tables in a 1 MiB scratch array compiled into
the library.  These tests call it through the C ABI and compare its output
with the regular dpred_flush_bucket (given a workspace) on the same inputs,
bit for bit, on two calls in a row, with a bucket large enough (300 tasks)
that its task table really goes through the scratch array.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import zero_collectives_gb300 as zc
from datagen import BF16, NORMAL, workloads
from tests.gpu_util import device_matrix

pytestmark = pytest.mark.gpu


def _case():
    world = 8
    sizes = np.array([(i * 53) % 700 + 1 for i in range(300)], np.int64)
    tree = workloads.Tree([f"p{i}" for i in range(len(sizes))], sizes)
    layout = workloads.arrival_layout(tree, capacity=None)
    return world, tree, layout


def test_noalloc_matches_workspace_flush_on_two_calls():
    world, tree, layout = _case()
    b = layout.buckets[0]
    assert zc.flush_workspace_bytes(world, len(b.tasks)) > 0, "the task table must go through the scratch"
    om = zc.build_owner_map(world, [(None, tree.numel)], True)
    ws = torch.empty(zc.flush_workspace_bytes(world, len(b.tasks)), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((7, 8)):
        grads = device_matrix(world, tree.total, BF16, NORMAL, seed, sigma=1e-2)
        ref = zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
        new = zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
        p_ref = zc.flush_bucket(grads, b.tasks, om.owner, ref.dst_table(b.tasks), BF16, True, True, probe=True,
                                workspace=ws)
        p_new = zc.flush_bucket_noalloc(grads, b.tasks, om.owner, new.dst_table(b.tasks), BF16, True, True,
                                        probe=True)
        torch.cuda.synchronize()
        for r in range(world):
            assert torch.equal(ref.buf[r].view(torch.int16), new.buf[r].view(torch.int16)), f"call {call} rank {r}"
            delivered = sum(int(tree.numel[p]) for p in range(tree.n_params)
                            if om.owner[p] == r or (om.owner[p] < 0 and om.holder_lo[p] <= r <= om.holder_hi[p]))
            written = int((~torch.isnan(new.buf[r].float())).sum().item())
            assert written == delivered, f"call {call} rank {r}: {written} written, {delivered} delivered"
        assert p_new.kept_elems == p_ref.kept_elems and p_new.owner_elems == p_ref.owner_elems
    assert zc.device_status() == 0


def test_noalloc_rejects_a_plan_beyond_the_scratch():
    world = 64
    n_tasks = 4000   # 4000 * 32 + 64 * 4000 * 8 bytes > 1 MiB
    assert zc.flush_workspace_bytes(world, n_tasks) > (1 << 20)
    tasks = np.zeros(n_tasks, dtype=zc.TASK_DTYPE)
    tasks["param_id"] = np.arange(n_tasks)
    tasks["offset"] = np.arange(n_tasks)
    tasks["numel"] = 1
    grads = torch.zeros((world, n_tasks), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(zc.DpredError) as e:
        zc.flush_bucket_noalloc(grads, tasks, None, None, BF16)
    assert e.value.code == -3 and "at most" in str(e.value)
