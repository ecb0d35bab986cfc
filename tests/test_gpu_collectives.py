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


@pytest.mark.parametrize("form", [zc.AG_REGISTER, zc.AG_TMA1, zc.AG_TMA4, zc.AG_STAGED, zc.AG_SKEW, zc.AG_SKEW8K],
                         ids=["register", "tma1", "tma4", "staged", "skew", "skew8k"])
@pytest.mark.parametrize("N", [1, 3, 4, 8, 16])
@pytest.mark.parametrize("order", [0, 1])
def test_allgather_forms(form, N, order):
    """Every AllGather kernel form gives the oracle's bytes, on shards that are
    a whole number of 8/16 KB tiles, end in a short tile, or are too short for
    a tile (bf16 rows of 16-byte multiples take the bulk-copy forms)."""
    prev = zc.set_allgather_form(form)
    try:
        for dt, S in ((BF16, 8), (BF16, 4096 * 3), (BF16, 65536 + 8), (F32, 8192 + 4), (BF16, 3 * 65536)):
            x = device_matrix(N, S, dt, UNIFORM, 16 + S % 7)
            out = torch.full((N, N * S), float("nan"), dtype=TORCH_DT[dt], device="cuda")
            zc.allgather(x, out, order)
            want = oracle.allgather(datagen.host_matrix(N, S, dt, UNIFORM, 16 + S % 7), order)
            torch.cuda.synchronize()
            assert np.array_equal(to_bits(out), np_bits(want)), f"{dt} S={S}"
    finally:
        zc.set_allgather_form(prev)
    assert zc.device_status() == 0


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
    for order, form in ((0, zc.AG_AUTO), (1, zc.AG_AUTO), (0, zc.AG_TMA4), (1, zc.AG_STAGED), (0, zc.AG_REGISTER), (0, zc.AG_SKEW), (1, zc.AG_SKEW8K)):
        ag = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
        prev = zc.set_allgather_form(form)
        zc.allgather(rs, ag, order)
        zc.set_allgather_form(prev)
        torch.cuda.synchronize()
        for i in range(N):
            for c in range(N):
                src = c if order == 0 else (i - c) % N
                assert torch.equal(ag[i, c * S:(c + 1) * S].view(torch.int16), rs[src].view(torch.int16))
        del ag


@pytest.mark.parametrize("method", [0, 1, 2])
def test_fill_pattern_writes_every_byte(method):
    """The write-only fill (the HBM write-ceiling kernel) writes its pattern to
    exactly the bytes it is given: the guard words around the range keep
    their value."""
    for nbytes in (32, 4096 + 32, 16384 * 7 + 96, (1 << 24) + 64):
        buf = torch.full((nbytes // 4 + 16,), -1, dtype=torch.int32, device="cuda")
        body = buf[8:8 + nbytes // 4]
        zc.fill_pattern(body, pattern=0x12345678, method=method)
        torch.cuda.synchronize()
        assert bool((body == 0x12345678).all()), nbytes
        assert bool((buf[:8] == -1).all()) and bool((buf[8 + nbytes // 4:] == -1).all()), nbytes


def test_stream_mixed_writes_pattern_and_leaves_its_source():
    """The mixed-traffic ceiling kernel writes its pattern over exactly the
    destination bytes (guards intact) and never writes its source."""
    for rb, wb in ((16384 * 3 + 48, 16384 * 20 + 32), (1 << 20, 8 << 20), (0, 4096), (4096, 0)):
        src = torch.arange(max(rb // 4, 1), dtype=torch.int32, device="cuda")
        keep = src.clone()
        buf = torch.full((wb // 4 + 16,), -1, dtype=torch.int32, device="cuda")
        body = buf[8:8 + wb // 4]
        zc.stream_mixed(src, body, read_bytes=rb, write_bytes=wb)
        torch.cuda.synchronize()
        assert bool((body == 0x3F803F80).all()) and bool((buf[:8] == -1).all()) and bool((buf[8 + wb // 4:] == -1).all())
        assert torch.equal(src, keep)
    assert zc.device_status() == 0
