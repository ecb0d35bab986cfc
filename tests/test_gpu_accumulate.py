"""GPU parity of dpred_accumulate_microbatch against the CPU oracle: bit-exact
for the deferred path (same order of operations), within the reassociation
tolerance against the per-micro-batch all-reduce, and the full qwen3-0.6b
shaped W=4 x 8 micro-batch step on sampled columns."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, NORMAL, stream_id, workloads
from tests.gpu_util import TORCH_DT, device_matrix, to_bits

pytestmark = pytest.mark.gpu


def run(world, n, n_mb, g_dt, scale=1.0, offset=0, seed=4):
    """Deferred accumulation on the GPU (acc and g offset by `offset` elements
    from a 16-byte boundary to reach the scalar path) and in the oracle."""
    acc_store = torch.full((world * n + offset,), float("nan"), dtype=torch.float32, device="cuda")
    acc = acc_store[offset:].view(world, n)
    total = torch.empty(n, dtype=torch.float32, device="cuda")
    host_acc = np.full((world, n), np.nan, np.float32)
    host_total = None
    g_all = []
    for m in range(n_mb):
        gs = torch.empty(world * n + offset, dtype=TORCH_DT[g_dt], device="cuda")
        g = gs[offset:].view(world, n)
        datagen.fill_device(g.data_ptr(), world, n, n, g_dt, NORMAL, seed, stream_id(0, m), 1, 0, 1e-3,
                            torch.cuda.current_stream().cuda_stream)
        gh = datagen.host_matrix(world, n, g_dt, NORMAL, seed, stream0=stream_id(0, m), sigma=1e-3)
        g_all.append(gh)
        last = m == n_mb - 1
        zc.accumulate_microbatch(acc, g, first=(m == 0), finalize=last, scale=scale, total=total if last else None)
        host_total = oracle.accumulate(host_acc, gh, first=(m == 0), finalize=last, scale=scale)
        if not last:
            torch.cuda.synchronize()
            assert np.array_equal(to_bits(acc), host_acc.view(np.uint32)), f"accumulator after micro-batch {m}"
    torch.cuda.synchronize()
    return to_bits(total).view(np.float32), host_total, np.stack(g_all)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 5])
@pytest.mark.parametrize("g_dt", [F32, BF16])
@pytest.mark.parametrize("offset", [0, 1])
def test_deferred_bit_exact(world, g_dt, offset):
    n = 3 * 4096 + 37 if offset == 0 else 4096 * 2 + 3
    got, want, g = run(world, n, 4, g_dt, offset=offset)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    per_mb = oracle.reduce_each_microbatch(g).astype(np.float64)
    d = got.astype(np.float64)
    assert np.linalg.norm(d - per_mb) / np.linalg.norm(per_mb) <= 5e-5


def test_single_microbatch_and_scale():
    got, want, g = run(4, 10000, 1, F32, scale=0.125)
    assert np.array_equal(got, want)
    assert np.array_equal(got, (oracle.reduce_each_microbatch(g) * np.float32(0.125)).astype(np.float32))


def test_finalize_leaves_accumulator_unchanged():
    world, n = 4, 8192
    acc = device_matrix(world, n, F32, NORMAL, 1, sigma=1.0)
    before = acc.clone()
    g = device_matrix(world, n, F32, NORMAL, 2, sigma=1.0)
    total = torch.empty(n, dtype=torch.float32, device="cuda")
    zc.accumulate_microbatch(acc, g, first=False, finalize=True, total=total)
    torch.cuda.synchronize()
    assert torch.equal(acc.view(torch.int32), before.view(torch.int32))


def test_qwen3_full_size_sampled():
    """W=4 replicas, 8 micro-batches, n = 596,049,920 (the qwen3-0.6b tree),
    fp32 gradients regenerated on the device per micro-batch."""
    world, n_mb, seed, sigma = 4, 8, 4, 1e-3
    n = workloads.tree_qwen3_06b().total
    acc = torch.empty((world, n), dtype=torch.float32, device="cuda")
    g = torch.empty((world, n), dtype=torch.float32, device="cuda")
    total = torch.empty(n, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for m in range(n_mb):
        datagen.fill_device(g.data_ptr(), world, n, n, F32, NORMAL, seed, stream_id(0, m), 1, 0, sigma, s)
        last = m == n_mb - 1
        zc.accumulate_microbatch(acc, g, first=(m == 0), finalize=last, total=total if last else None)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    cols = np.unique(np.concatenate([[0, n - 1, n // 2], rng.integers(0, n, size=20000)])).astype(np.int64)
    gs = np.stack([np.stack([datagen.sample_host(np.full(len(cols), stream_id(r, m)), cols, F32, NORMAL, seed, sigma)
                             for r in range(world)]) for m in range(n_mb)])
    host_acc = np.empty((world, len(cols)), np.float32)
    for m in range(n_mb):
        want = oracle.accumulate(host_acc, np.ascontiguousarray(gs[m]), first=(m == 0), finalize=(m == n_mb - 1))
    got = to_bits(total[torch.from_numpy(cols).cuda()]).view(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    per_mb = oracle.reduce_each_microbatch(gs).astype(np.float64)
    assert np.linalg.norm(got.astype(np.float64) - per_mb) / np.linalg.norm(per_mb) <= 5e-5


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("offset", [0, 1])
def test_checkpoint_save_restore_bit_exact(world, offset):
    n = 4096 * 3 + (0 if offset == 0 else 5)
    store = torch.empty(world * n + offset, dtype=torch.float32, device="cuda")
    acc = store[offset:].view(world, n)
    datagen.fill_device(acc.data_ptr(), world, n, n, F32, NORMAL, 11, 0, 1, 0, 1e-3,
                        torch.cuda.current_stream().cuda_stream)
    tstore = torch.empty(n + offset, dtype=torch.float32, device="cuda")
    total = tstore[offset:]
    zc.accumulator_save(acc, total)
    host_acc = datagen.host_matrix(world, n, F32, NORMAL, 11, sigma=1e-3)
    want = oracle.accumulator_save(host_acc)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(total), want.view(np.uint32))
    zc.accumulator_restore(acc, total)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(acc), oracle.accumulator_restore(want, world).view(np.uint32))


def test_mid_step_checkpoint_round_trip_on_gpu():
    """Accumulate 3 of 8 micro-batches, save, restore, finish: bit-identical to
    the oracle doing the same, and within the reassociation tolerance of the
    uninterrupted step."""
    world, n, n_mb, cut = 4, 20000, 8, 3
    s = torch.cuda.current_stream().cuda_stream
    acc = torch.empty((world, n), dtype=torch.float32, device="cuda")
    g = torch.empty((world, n), dtype=torch.float32, device="cuda")
    total = torch.empty(n, dtype=torch.float32, device="cuda")
    host_acc = np.empty((world, n), np.float32)
    gs = []
    for m in range(n_mb):
        datagen.fill_device(g.data_ptr(), world, n, n, F32, NORMAL, 4, stream_id(0, m), 1, 0, 1e-3, s)
        gh = datagen.host_matrix(world, n, F32, NORMAL, 4, stream0=stream_id(0, m), sigma=1e-3)
        gs.append(gh)
        last = m == n_mb - 1
        zc.accumulate_microbatch(acc, g, first=(m == 0), finalize=last, total=total if last else None)
        want = oracle.accumulate(host_acc, gh, first=(m == 0), finalize=last)
        if m == cut - 1:
            zc.accumulator_save(acc, total)
            zc.accumulator_restore(acc, total)
            host_acc = oracle.accumulator_restore(oracle.accumulator_save(host_acc), world)
    torch.cuda.synchronize()
    got = to_bits(total).view(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    straight = np.empty((world, n), np.float32)
    for m in range(n_mb):
        ref = oracle.accumulate(straight, gs[m], first=(m == 0), finalize=(m == n_mb - 1))
    d, r = got.astype(np.float64), ref.astype(np.float64)
    assert np.linalg.norm(d - r) / np.linalg.norm(r) <= 5e-5
