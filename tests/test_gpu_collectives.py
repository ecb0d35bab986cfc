"""GPU parity of dpred_reduce_scatter and dpred_allgather (canonical and ring
order) against the CPU oracle, RS followed by AG against the AllReduce form of
the flush, and the 1 GiB bf16 layouts at N = 4 and 8."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, UNIFORM, workloads
from tests.gpu_util import TORCH_DT, device_matrix, np_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[zc.PATH_LDG, zc.PATH_TMA], ids=["ldg", "tma"], autouse=True)
def flush_path(request):
    """Run every test with both flush kernel families (results must be bit-identical)."""
    prev = zc.set_flush_path(request.param)
    yield request.param
    zc.set_flush_path(prev)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("in_dt,out_dt", [(BF16, BF16), (F32, F32), (BF16, F32)])
@pytest.mark.parametrize("pre_div", [False, True])
def test_reduce_scatter(N, in_dt, out_dt, pre_div):
    for S in (1, 7, 4096 * 3 + 5):
        M = N * S
        x = device_matrix(N, M, in_dt, UNIFORM, 5)
        out = torch.full((N, S), float("nan"), dtype=TORCH_DT[out_dt], device="cuda")
        zc.reduce_scatter(x, out, pre_div)
        want = oracle.reduce_scatter(datagen.host_matrix(N, M, in_dt, UNIFORM, 5), pre_div, out_dt)
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(out), np_bits(want))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_allgather(N, order, dt):
    for S in (1, 5, 8192 + 3, 65536):
        x = device_matrix(N, S, dt, UNIFORM, 6)
        out = torch.full((N, N * S), float("nan"), dtype=TORCH_DT[dt], device="cuda")
        zc.allgather(x, out, order)
        want = oracle.allgather(datagen.host_matrix(N, S, dt, UNIFORM, 6), order)
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(out), np_bits(want))


@pytest.mark.parametrize("N", [2, 4, 8])
def test_reduce_scatter_then_allgather_is_allreduce(N):
    S = 3 * 8192 + 8
    M = N * S
    x = device_matrix(N, M, BF16, UNIFORM, 7)
    ar = x.clone()
    tasks = np.zeros(1, dtype=zc.TASK_DTYPE)
    tasks["numel"] = M
    zc.flush_bucket(ar, tasks, None, None, BF16, pre_div=False, reduce_to_owner=False)  # AllReduce in place
    rs = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
    ag = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    zc.reduce_scatter(x, rs)
    zc.allgather(rs, ag, 0)
    torch.cuda.synchronize()
    assert torch.equal(ag.view(torch.int16), ar.view(torch.int16))


@pytest.mark.parametrize("N", [4, 8])
def test_one_gib_layouts(N):
    M = 1 << 29
    S = M // N
    x = device_matrix(N, M, BF16, UNIFORM, 5)
    rs = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
    zc.reduce_scatter(x, rs)
    torch.cuda.synchronize()
    rng = np.random.default_rng(N)
    cols = np.unique(np.concatenate([[0, M - 1, S - 1, S], rng.integers(0, M, size=20000)])).astype(np.int64)
    xs = np.stack([datagen.sample_host(np.full(len(cols), j), cols, BF16, UNIFORM, 5) for j in range(N)])
    want = oracle.reduce_rows(xs, pre_div=False)
    got = to_bits(rs.view(-1)[torch.from_numpy(cols).cuda()])
    assert np.array_equal(got, want)
    del x
    for order in (0, 1):
        ag = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
        zc.allgather(rs, ag, order)
        torch.cuda.synchronize()
        for i in range(N):
            for c in range(N):
                src = c if order == 0 else (i - c) % N
                assert torch.equal(ag[i, c * S:(c + 1) * S].view(torch.int16), rs[src].view(torch.int16))
        del ag
