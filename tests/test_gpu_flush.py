"""GPU parity of dpred_flush_bucket against the CPU oracle (bit-exact).

The tiny workload (W=4, 16 parameters of 1..4096 elements, straddlers), a
sweep of world sizes / dtypes / straddler counts / excluded groups with both
the 16-byte vector path and the scalar path, the in-place form, the
workspace plan, and the full 402.8M-parameter W=8 flush in the configuration
the bench times (sampled outputs checked one by one)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import zero_collectives_gb300 as zc
from datagen import BF16, F32, NORMAL, workloads
from tests.gpu_util import TORCH_DT, device_matrix, np_bits, oracle_flush, to_bits
from tests.helpers import holder_sets, is_sentinel, oracle_dst

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[zc.PATH_LDG, zc.PATH_TMA], ids=["ldg", "tma"], autouse=True)
def flush_path(request):
    """Run every test with both flush kernel families (results must be bit-identical)."""
    prev = zc.set_flush_path(request.param)
    yield request.param
    zc.set_flush_path(prev)

GUARD = 16  # canary elements before and after every destination


class SlotBuffers:
    """One NaN-filled CUDA buffer per (rank, held parameter) with GUARD canary
    elements on each side; `shift` moves the destination by whole elements
    (shift 'co' keeps it co-aligned with its source, 'mis' breaks that)."""

    def __init__(self, world, tasks, holders, out_dt, in_dt, mode):
        vec = 8 if in_dt == BF16 else 4
        self.world, self.tasks = world, tasks
        self.buf, self.off = {}, {}
        ptrs = []
        for r in range(world):
            for task in tasks:
                p, off, n = int(task["param_id"]), int(task["offset"]), int(task["numel"])
                if r not in holders[p]:
                    ptrs.append(0)
                    continue
                shift = off % vec + (1 if mode == "mis" else 0)
                b = torch.full((n + 2 * GUARD + vec,), float("nan"), dtype=TORCH_DT[out_dt], device="cuda")
                self.buf[(r, p)] = b
                self.off[(r, p)] = GUARD + shift
                ptrs.append(b.data_ptr() + (GUARD + shift) * b.element_size())
        self.table = zc.DstTable(world, len(tasks), ptrs)

    def check_against(self, oracle_dst, tasks, out_dt):
        """Delivered slots equal the oracle bit for bit; the rest and the guards stay NaN."""
        for t, task in enumerate(tasks):
            p, n = int(task["param_id"]), int(task["numel"])
            for r in range(self.world):
                o = oracle_dst[r][t]
                if o is None:
                    assert (r, p) not in self.buf
                    continue
                b = self.buf[(r, p)]
                s = self.off[(r, p)]
                got = to_bits(b)
                isn = torch.isnan(b.float()).cpu().numpy()
                assert isn[:s].all() and isn[s + n:].all(), f"canary overwritten at rank {r} param {p}"
                if np.all(is_sentinel(o, out_dt == BF16)):
                    assert isn[s:s + n].all(), f"non-delivered buffer written at rank {r} param {p}"
                else:
                    assert np.array_equal(got[s:s + n], np_bits(o)), f"rank {r} param {p}"


def run_case(world, groups, in_dt, out_dt, pre_div, rto, mode="co", capacity=None, seed=21, ld_pad=0, sigma=1e-2):
    numel = np.concatenate([np.asarray(g[1], np.int64) for g in groups])
    tree = workloads.Tree([f"p{i}" for i in range(len(numel))], numel)
    layout = workloads.arrival_layout(tree, capacity=capacity)
    row = tree.total
    ld = row + ld_pad
    grads = device_matrix(world, row, in_dt, NORMAL, seed, sigma=sigma, ld=ld)
    host = datagen.host_matrix(world, row, in_dt, NORMAL, seed, sigma=sigma)
    zgroups = [(None if list(g[0]) == list(range(world)) else g[0], g[1]) for g in groups]
    om = zc.build_owner_map(world, zgroups, rto)
    holders = holder_sets(om.holder_lo, om.holder_hi)
    for b in layout.buckets:
        sb = SlotBuffers(world, b.tasks, holders, out_dt, in_dt, mode)
        wsb = zc.flush_workspace_bytes(world, len(b.tasks))  # plans beyond the inline limits (many ranks)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
        probe = zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, om.owner, sb.table, out_dt, pre_div,
                                rto, checked=True, probe=True, workspace=ws)
        sub = np.ascontiguousarray(host[:, b.start:b.start + b.size])
        odst, oom, oprobe = oracle_flush(world, sub, b.tasks, numel, groups, out_dt, pre_div, rto, tree.n_params)
        assert np.array_equal(oom["owner"], om.owner)
        torch.cuda.synchronize()
        sb.check_against(odst, b.tasks, out_dt)
        assert (probe.tasks, probe.reduced_elems, probe.owner_tasks, probe.owner_elems) == \
            (oprobe["tasks"], oprobe["reduced_elems"], oprobe["owner_tasks"], oprobe["owner_elems"])
        assert probe.kept_elems == oprobe["kept_elems"]
    assert zc.device_status() == 0


@pytest.mark.parametrize("rto", [True, False])
@pytest.mark.parametrize("out_dt", [BF16, F32])
@pytest.mark.parametrize("mode", ["co", "mis"])
def test_tiny_workload(rto, out_dt, mode):
    world = 4
    tree = workloads.tree_tiny(seed=1)
    run_case(world, [(list(range(world)), tree.numel)], BF16, out_dt, True, rto, mode=mode, seed=2)


@pytest.mark.parametrize("world", [*range(2, 18), 24, 32, 33, 48, 64])  # every unrolled size, then the generic loops
@pytest.mark.parametrize("in_dt,out_dt", [(BF16, BF16), (F32, F32), (BF16, F32), (F32, BF16)])
def test_sweep_world_dtype_straddlers(world, in_dt, out_dt):
    rng = np.random.default_rng(world * 7 + in_dt * 3 + out_dt)
    for straddlers in sorted({0, world // 2, world - 1}):
        elems = int(rng.integers(3, 9)) * 8192 * world + int(rng.integers(0, 999))  # several units + ragged tail
        tree = workloads.straddle_tree(world, elems, straddlers)
        groups = [(list(range(world)), tree.numel)]
        if world >= 4:
            groups.append((list(range(world // 2)), np.array([777, 4096, 33], np.int64)))  # excluded group
        for pre_div, rto in ((True, True), (False, False)):
            run_case(world, groups, in_dt, out_dt, pre_div, rto, mode="co", seed=30 + straddlers)
    run_case(world, [(list(range(world)), workloads.straddle_tree(world, 5000 * world + 7, world - 1).numel)],
             in_dt, out_dt, True, True, mode="mis", seed=41, ld_pad=5)


def test_many_tasks_use_the_workspace_plan():
    world = 8
    sizes = np.array([(i * 37) % 500 + 1 for i in range(300)], np.int64)
    assert zc.flush_workspace_bytes(world, 300) > 0
    tree = workloads.Tree([f"p{i}" for i in range(300)], sizes)
    layout = workloads.arrival_layout(tree, capacity=None)
    b = layout.buckets[0]
    grads = device_matrix(world, tree.total, BF16, NORMAL, 7, sigma=1e-2)
    host = datagen.host_matrix(world, tree.total, BF16, NORMAL, 7, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, sizes)], False)
    holders = holder_sets(om.holder_lo, om.holder_hi)
    sb = SlotBuffers(world, b.tasks, holders, BF16, BF16, "co")
    ws = torch.empty(zc.flush_workspace_bytes(world, len(b.tasks)), dtype=torch.uint8, device="cuda")
    with pytest.raises(zc.DpredError):
        zc.flush_bucket(grads, b.tasks, om.owner, sb.table, BF16, True, False)  # no workspace given
    zc.flush_bucket(grads, b.tasks, om.owner, sb.table, BF16, True, False, workspace=ws)
    odst, _, _ = oracle_flush(world, host, b.tasks, sizes, [(list(range(world)), sizes)], BF16, True, False, 300)
    torch.cuda.synchronize()
    sb.check_against(odst, b.tasks, BF16)


@pytest.mark.parametrize("rto", [True, False])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_in_place(rto, dt):
    world = 8
    tree = workloads.straddle_tree(world, 40000 * world + 13, 5)
    layout = workloads.arrival_layout(tree, capacity=None)
    b = layout.buckets[0]
    grads = device_matrix(world, tree.total, dt, NORMAL, 9, sigma=1e-2)
    host = datagen.host_matrix(world, tree.total, dt, NORMAL, 9, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, tree.numel)], rto)
    probe = zc.flush_bucket(grads, b.tasks, om.owner, None, dt, True, rto, probe=True)
    oprobe = oracle.flush(world, host, b.tasks, om.owner, tree.n_params, None, dt, True, rto)
    assert np.array_equal(to_bits(grads), np_bits(host))
    assert probe.kept_elems == oprobe["kept_elems"]


@pytest.mark.parametrize("world", [2, 3, 4, 5, 6, 7, 8, 9, 12, 13, 16, 24, 64])
def test_every_bf16_pattern(world):
    """All 65,536 bf16 bit patterns (subnormals, signed zeros, infinities,
    NaNs), rotated differently in every replica row, plus a block of columns
    drawn only from subnormals and the smallest normals, so that pre-divided
    terms sit at the bottom of the fp32 range.  In-place AllReduce form,
    pre-division on: every row must equal the oracle bit for bit (a NaN only
    has to stay NaN: the kernel's conversion returns a canonical NaN)."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    tiny = np.concatenate([np.arange(0x0000, 0x0100), np.arange(0x8000, 0x8100)]).astype(np.uint16)
    rng = np.random.default_rng(world)
    n = len(pats) + 4096
    host = np.empty((world, n), np.uint16)
    for r in range(world):
        host[r, :len(pats)] = np.roll(pats, r * 7919)
        host[r, len(pats):] = rng.choice(tiny, 4096)
    grads = torch.from_numpy(host.view(np.int16).copy()).cuda().view(torch.bfloat16)
    tasks = np.zeros(1, dtype=zc.TASK_DTYPE)
    tasks["numel"] = n
    zc.flush_bucket(grads, tasks, None, None, BF16, True, False)
    oracle.flush(world, host, tasks, None, 1, None, BF16, True, False)
    torch.cuda.synchronize()
    got = to_bits(grads)

    def nan(b):
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)

    same = (got == host) | (nan(got) & nan(host))
    assert same.all(), f"{int((~same).sum())} elements differ, first at {np.argwhere(~same)[0]}"
    assert zc.device_status() == 0


@pytest.mark.parametrize("world", [3, 6, 7, 12, 13, 24])
def test_fp32_terms_at_the_bottom_of_the_range(world):
    """fp32 terms divided by a rank count that is not a power of two: the
    kernels' division-free quotient leaves tiny terms (0 < |x| < 2^-120) to
    IEEE division.  Rows mix subnormals, the normals around 2^-120, signed
    zeros, ordinary values, infinities and NaNs, so that the vector path meets
    tiny terms in some vectors and none in others; every output must equal the
    oracle bit for bit (a NaN only has to stay NaN)."""
    rng = np.random.default_rng(100 + world)
    n = 64 * 1024 + 13
    pools = [
        rng.integers(1, 0x00800000, 4096, dtype=np.uint32),                  # subnormals
        rng.integers(0x03000000, 0x04000000, 4096, dtype=np.uint32),         # around 2^-120
        np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000], np.uint32),
        rng.integers(0x38000000, 0x3F800000, 4096, dtype=np.uint32),         # ordinary values
    ]
    host = np.empty((world, n), np.uint32)
    for r in range(world):
        kind = rng.integers(0, 8, n)
        vals = np.where(kind == 0, rng.choice(pools[0], n),
                        np.where(kind == 1, rng.choice(pools[1], n),
                                 np.where(kind == 2, rng.choice(pools[2], n), rng.choice(pools[3], n))))
        host[r] = vals | (rng.integers(0, 2, n, dtype=np.uint32) << 31)
        host[r, : n // 3] = rng.choice(pools[3], n // 3)                      # a stretch without tiny terms
    grads = torch.from_numpy(host.view(np.int32).copy()).cuda().view(torch.float32)
    tasks = np.zeros(1, dtype=zc.TASK_DTYPE)
    tasks["numel"] = n
    zc.flush_bucket(grads, tasks, None, None, F32, True, False)
    want = host.view(np.float32).copy()
    oracle.flush(world, want, tasks, None, 1, None, F32, True, False)
    torch.cuda.synchronize()
    got = to_bits(grads)
    wb = want.view(np.uint32)

    def nan(b):
        return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x7FFFFF) != 0)

    same = (got == wb) | (nan(got) & nan(wb))
    assert same.all(), f"{int((~same).sum())} elements differ, first at {np.argwhere(~same)[0]}"
    assert zc.device_status() == 0


def test_identical_replicas_reproduce_exactly():
    """The DeepSpeed issue's exactness check: identical input on every rank
    reproduces the input exactly (bf16, pre-division by a power of two)."""
    world = 8
    tree = workloads.tree_tiny(seed=1)
    row = device_matrix(1, tree.total, BF16, NORMAL, 3, sigma=1e-2)
    grads = row.repeat(world, 1).contiguous()
    layout = workloads.arrival_layout(tree, capacity=None)
    om = zc.build_owner_map(world, [(None, tree.numel)])
    zc.flush_bucket(grads, layout.buckets[0].tasks, om.owner, None, BF16, True, True)
    for t in layout.buckets[0].tasks:
        o, n = int(t["offset"]), int(t["numel"])
        p = int(t["param_id"])
        r = om.owner[p] if om.owner[p] >= 0 else 0
        assert torch.equal(grads[r, o:o + n].view(torch.int16), row[0, o:o + n].view(torch.int16))


@pytest.mark.parametrize("path", ["calls", "executor"])
def test_402m_w8_full_size_sampled(path):
    """The full 402.8M-parameter W=8 bf16 flush (7 buckets, reduce-to-owner)
    in the configurations the bench times: 7 dpred_flush_bucket calls with the
    probe counters and the overlap promise (checked on the second step, whose
    plans come from the plan cache, after the buffers are refilled with NaN),
    and the executor's one-call step."""
    world, sigma, seed = 8, 1e-3, 3
    tree = workloads.tree_402m()
    layout = workloads.arrival_layout(tree)
    grads = device_matrix(world, tree.total, BF16, NORMAL, seed, sigma=sigma)
    ex = zc.Zero1Executor(world, tree.numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets],
                          torch.bfloat16, fill=float("nan"))
    if path == "executor":
        probes = ex.flush_all(grads, probe=True)
    else:
        calls = [(grads[:, s0:s0 + size], t, tab) for (s0, t), size, tab in zip(ex.buckets, ex.sizes, ex.tables)]
        for step in range(2):
            if step == 1:
                torch.cuda.synchronize()
                for buf in ex.grad.buf:
                    buf.fill_(float("nan"))
            probes = [zc.flush_bucket(g, t, ex.omap.owner, tab, BF16, True, True, probe=True, flush_index=i,
                                      overlap=True) for i, (g, t, tab) in enumerate(calls)]
    torch.cuda.synchronize()
    assert zc.device_status() == 0
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)])
    assert np.array_equal(om["owner"], ex.omap.owner)
    # every delivered slot fully written, nothing else
    for r in range(world):
        delivered = sum(int(tree.numel[p]) for p in range(tree.n_params)
                        if om["owner"][p] == r or (om["owner"][p] < 0 and om["holder_lo"][p] <= r <= om["holder_hi"][p]))
        written = int((~torch.isnan(ex.grad.buf[r].float())).sum().item())
        assert written == delivered, f"rank {r}: {written} written, {delivered} delivered"
    # sampled values, one by one against the oracle
    rng = np.random.default_rng(0)
    picks = []
    for p in range(tree.n_params):
        n = int(tree.numel[p])
        ks = {0, n - 1} | set(int(v) for v in rng.integers(0, n, size=24))
        picks += [(p, k) for k in sorted(ks)]
    P = np.array([p for p, _ in picks])
    K = np.array([k for _, k in picks])
    cols = layout.row_offset[P] + K
    x = np.stack([datagen.sample_host(np.full(len(cols), r), cols, BF16, NORMAL, seed, sigma) for r in range(world)])
    want = oracle.reduce_rows(x, pre_div=True)
    for r in range(world):
        sel = [i for i, p in enumerate(P) if om["owner"][p] == r or
               (om["owner"][p] < 0 and om["holder_lo"][p] <= r <= om["holder_hi"][p])]
        idx = torch.tensor([ex.grad.slot[r][int(P[i])] + int(K[i]) for i in sel], device="cuda")
        got = to_bits(ex.grad.buf[r][idx])
        assert np.array_equal(got, want[sel]), f"rank {r}"
    # probe totals
    assert sum(p.owner_elems for p in probes) == 295_798_784
    assert sum(p.reduced_elems for p in probes) == tree.total


@pytest.mark.parametrize("world,dt", [(2, BF16), (16, BF16), (8, F32)])
def test_sweep_1gb_per_replica_sampled(world, dt):
    """The largest sweep case (1 GB per replica row) in the layout the sweep
    times: one bucket whose W-1 interior partition boundaries all fall inside
    a parameter, plus a 3-parameter group on a smaller communicator (AllReduce
    to every rank), flushed through the executor.  Every delivered slot is
    fully written and nothing else; sampled values (both ends of every
    parameter, the elements around every partition boundary and random ones)
    equal the oracle bit for bit."""
    esize = 2 if dt == BF16 else 4
    seed, sigma = 6, 1e-3
    tree = workloads.straddle_tree(world, (1 << 30) // esize, world - 1, pieces=2)
    ex_sizes = np.array([96, 64, 32], np.int64)
    numel = np.concatenate([tree.numel, ex_sizes])
    full = workloads.Tree([f"p{i}" for i in range(len(numel))], numel)
    layout = workloads.arrival_layout(full, capacity=None)
    sub = list(range(max(1, world // 2)))
    grads = device_matrix(world, full.total, dt, NORMAL, seed, sigma=sigma)
    ex = zc.Zero1Executor(world, numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets], TORCH_DT[dt],
                          groups=[(None, tree.numel), (sub, ex_sizes)], fill=float("nan"))
    ex.flush_all(grads)
    torch.cuda.synchronize()
    assert zc.device_status() == 0
    om = oracle.owner_map(world, [(list(range(world)), tree.numel), (sub, ex_sizes)])
    assert np.array_equal(om["owner"], ex.omap.owner)
    holders = holder_sets(om["holder_lo"], om["holder_hi"])
    delivered = [[p for p in range(full.n_params) if (om["owner"][p] == r or (om["owner"][p] < 0 and r in holders[p]))]
                 for r in range(world)]
    for r in range(world):
        want = sum(int(numel[p]) for p in delivered[r])
        written = int((~torch.isnan(ex.grad.buf[r].float())).sum().item())
        assert written == want, f"rank {r}: {written} written, {want} delivered"
    del grads
    # samples: parameter ends, +-2 elements around every partition boundary, random
    rng = np.random.default_rng(world)
    T = int(tree.numel.sum())
    part = -(-T // world)
    flat0 = np.concatenate([[0], np.cumsum(numel)[:-1]])
    picks = set()
    for p in range(full.n_params):
        n = int(numel[p])
        picks |= {(p, 0), (p, n - 1)} | {(p, int(k)) for k in rng.integers(0, n, size=16)}
    for b in range(1, world):
        for f in range(b * part - 2, b * part + 2):
            p = int(np.searchsorted(flat0[:tree.n_params], f, side="right") - 1)
            if 0 <= f - flat0[p] < numel[p]:
                picks.add((p, int(f - flat0[p])))
    picks = sorted(picks)
    P = np.array([p for p, _ in picks])
    K = np.array([k for _, k in picks])
    cols = layout.row_offset[P] + K
    x = np.stack([datagen.sample_host(np.full(len(cols), r), cols, dt, NORMAL, seed, sigma) for r in range(world)])
    want = np_bits(oracle.reduce_rows(x, pre_div=True))
    for r in range(world):
        sel = [i for i, p in enumerate(P) if p in set(delivered[r])]
        idx = torch.tensor([ex.grad.slot[r][int(P[i])] + int(K[i]) for i in sel], device="cuda")
        got = to_bits(ex.grad.buf[r][idx])
        assert np.array_equal(got, want[sel]), f"rank {r}"
    ex.close()


def test_indices_beyond_int32():
    """A task longer than 2^31 elements and a task that starts past element
    2^31 of its row: every 64-bit index path (unit search, vector and scalar
    offsets, destinations) is exercised.  W=2 bf16, 8.6 GB of gradients;
    sampled elements against the oracle, the ends of every destination and
    the canaries around them checked exactly."""
    world, seed, sigma = 2, 41, 1e-2
    big = (1 << 31) + 11                      # numel above INT32_MAX, starts unaligned (head of 3)
    off1 = (1 << 31) + 100                    # second task starts past 2^31
    n1 = 3 * (1 << 20) - 77                   # ragged tail
    ld = off1 + n1 + 29
    grads = device_matrix(world, ld, BF16, NORMAL, seed, sigma=sigma)
    tasks = np.zeros(2, dtype=zc.TASK_DTYPE)
    tasks[0] = (0, 0, 5, big)
    tasks[1] = (1, 0, off1, n1)
    owner = np.array([1, -1], np.int32)       # param 0 reduced to rank 1, param 1 to both ranks
    g = 8
    b0 = torch.full((big + 2 * g,), float("nan"), dtype=torch.bfloat16, device="cuda")
    b1 = [torch.full((n1 + 2 * g,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    table = zc.DstTable(world, 2, [0, b1[0][g:].data_ptr(), b0[g:].data_ptr(), b1[1][g:].data_ptr()])
    pr = zc.flush_bucket(grads, tasks, owner, table, BF16, True, True, probe=True)
    torch.cuda.synchronize()
    assert zc.device_status() == 0
    assert pr.reduced_elems == big + n1 and pr.owner_elems == big
    rng = np.random.default_rng(7)

    def check(buf, off, n, picks):
        ks = np.array(sorted(set(int(k) for k in picks if 0 <= k < n)), np.int64)
        cols = off + ks
        x = np.stack([datagen.sample_host(np.full(len(cols), r), cols, BF16, NORMAL, seed, sigma) for r in range(world)])
        want = oracle.reduce_rows(x, pre_div=True)
        got = to_bits(buf[g + torch.from_numpy(ks).cuda()])
        assert np.array_equal(got, np_bits(want))
        assert torch.isnan(buf[:g].float()).all() and torch.isnan(buf[g + n:].float()).all()

    edge = [0, 1, 2, 3, 4, 5, 6, 7, 8]
    near = [(1 << 31) - 5 - d for d in range(-12, 12)]       # task-relative positions around row element 2^31
    check(b0, 5, big, edge + near + [big - 1 - d for d in range(16)] + list(rng.integers(0, big, 400)))
    for r in range(world):
        check(b1[r], off1, n1, edge + [n1 - 1 - d for d in range(16)] + list(rng.integers(0, n1, 200)))
    # no element of the long destination was left unwritten
    assert not torch.isnan(b0[g:g + big].float()).any()


def test_plan_cache_never_serves_a_stale_plan():
    """dpred_flush_bucket reuses the validated plan of a repeated call.  A call
    whose owner values, task table (changed in place, same arrays) or
    destination table differ in any byte must get its own plan: every result
    equals the oracle for that call's inputs, and buffers of an earlier table
    are left alone."""
    world, seed = 4, 31
    tree = workloads.tree_tiny(seed=1)
    b = workloads.arrival_layout(tree, capacity=None).buckets[0]
    grads = device_matrix(world, tree.total, BF16, NORMAL, seed, sigma=1e-2)
    host = datagen.host_matrix(world, tree.total, BF16, NORMAL, seed, sigma=1e-2)
    everyone = [set(range(world)) for _ in range(tree.n_params)]  # every rank has a buffer
    owner = zc.build_owner_map(world, [(None, tree.numel)], True).owner.copy()
    tasks = b.tasks.copy()

    def run(sb, label):
        probe = zc.flush_bucket(grads, tasks, owner, sb.table, BF16, True, True, probe=True)
        odst = oracle_dst(world, tasks, everyone, True)
        oprobe = oracle.flush(world, host.copy(), tasks, owner, tree.n_params, odst, BF16, True, True)
        torch.cuda.synchronize()
        sb.check_against(odst, tasks, BF16)
        assert probe.kept_elems == oprobe["kept_elems"], label
        assert (probe.owner_tasks, probe.owner_elems) == (oprobe["owner_tasks"], oprobe["owner_elems"]), label

    def refill(sb):
        torch.cuda.synchronize()
        for buf in sb.buf.values():
            buf.fill_(float("nan"))

    sb = SlotBuffers(world, tasks, everyone, BF16, BF16, "co")
    run(sb, "first call")
    refill(sb)
    run(sb, "the same call again")
    owned = owner >= 0
    assert owned.any()
    owner[owned] = (owner[owned] + 1) % world          # every owned parameter moves to the next rank
    refill(sb)
    run(sb, "owners changed in place")
    tasks["numel"][0] -= 1                              # the first task shrinks, same array
    refill(sb)
    run(sb, "task table changed in place")
    sb2 = SlotBuffers(world, tasks, everyone, BF16, BF16, "co")
    refill(sb)
    run(sb2, "new destination table")
    torch.cuda.synchronize()
    assert all(bool(torch.isnan(buf.float()).all()) for buf in sb.buf.values()), "old destinations written"
    assert zc.device_status() == 0


@pytest.mark.parametrize("world,in_dt", [(16, BF16), (24, BF16), (24, F32), (40, BF16), (64, BF16), (48, F32)])
def test_overlapped_calls_match_plain_calls_at_many_ranks(world, in_dt):
    """Consecutive flushes with the overlap promise at sizes whose kernels
    launch one CTA per work unit (W=16, the generic loop, the chunk-8 loop at
    powers of two) or keep a persistent grid (the chunk-8 loop at other
    sizes): every bucket's bits equal those of plain, serialised calls (which
    test_sweep_world_dtype_straddlers checks against the oracle at these
    sizes)."""
    dt = TORCH_DT[in_dt]
    tree = workloads.straddle_tree(world, 20000 * world + 3, world - 1, pieces=3)
    layout = workloads.arrival_layout(tree, capacity=tree.total // 3)
    assert len(layout.buckets) >= 3
    grads = device_matrix(world, tree.total, in_dt, NORMAL, 12, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, tree.numel)], True)
    bufs = [zc.GradBuffers(world, om, tree.numel, layout.row_offset, dt, fill=float("nan")) for _ in range(2)]
    for buf, overlap in zip(bufs, (False, True)):
        for b in layout.buckets:
            wsb = zc.flush_workspace_bytes(world, len(b.tasks))
            ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
            zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, om.owner, buf.dst_table(b.tasks), in_dt,
                            overlap=overlap, workspace=ws)
    torch.cuda.synchronize()
    bits = torch.int16 if in_dt == BF16 else torch.int32
    for r in range(world):
        assert torch.equal(bufs[0].buf[r].view(bits), bufs[1].buf[r].view(bits)), f"rank {r}"
    assert zc.device_status() == 0


def test_flush_bucket_call_paths_agree(monkeypatch):
    """zc.flush_bucket goes through the CPython module where it is built;
    forced onto ctypes, the same buckets give the same bits and probe
    counters."""
    if zc._fast_call_module() is None:
        pytest.skip("the CPython call module is not built on this host (no Python headers)")
    world = 8
    tree = workloads.straddle_tree(world, 30000 * world + 5, 5, pieces=3)
    layout = workloads.arrival_layout(tree, capacity=tree.total // 2)
    grads = device_matrix(world, tree.total, BF16, NORMAL, 9, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, tree.numel)], True)
    bufs = [zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
            for _ in range(2)]
    probes = []
    for k, buf in enumerate(bufs):
        if k == 1:
            monkeypatch.setattr(zc, "_FC", None)
            monkeypatch.setattr(zc, "_fast_call_module", lambda: None)
        probes.append([zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, om.owner, buf.dst_table(b.tasks),
                                       BF16, probe=True, flush_index=i) for i, b in enumerate(layout.buckets)])
    torch.cuda.synchronize()
    for r in range(world):
        assert torch.equal(bufs[0].buf[r].view(torch.int16), bufs[1].buf[r].view(torch.int16)), f"rank {r}"
    assert probes[0] == probes[1]
    assert [p.flush_index for p in probes[0]] == list(range(len(layout.buckets)))
    assert zc.device_status() == 0


@pytest.mark.parametrize("fast", [True, False], ids=["cpython", "ctypes"])
def test_prepared_call_matches_flush_bucket(fast):
    """zc.BucketFlush marshals a bucket's arguments once; every call gives the
    bits and probe counters of the plain call, step after step, with and
    without the overlap promise, through either call path."""
    if fast and zc._fast_call_module() is None:
        pytest.skip("the CPython call module is not built on this host (no Python headers)")
    world = 8
    tree = workloads.straddle_tree(world, 30000 * world + 5, 5, pieces=3)
    layout = workloads.arrival_layout(tree, capacity=tree.total // 2)
    grads = device_matrix(world, tree.total, BF16, NORMAL, 8, sigma=1e-2)
    om = zc.build_owner_map(world, [(None, tree.numel)], True)
    want = zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    got = zc.GradBuffers(world, om, tree.numel, layout.row_offset, torch.bfloat16, fill=float("nan"))
    probes_want = [zc.flush_bucket(grads[:, b.start:b.start + b.size], b.tasks, om.owner, want.dst_table(b.tasks),
                                   BF16, probe=True) for b in layout.buckets]
    calls = [zc.BucketFlush(grads[:, b.start:b.start + b.size], b.tasks, om.owner, got.dst_table(b.tasks),
                            overlap=overlap, fast=fast) for b, overlap in zip(layout.buckets, (False, True, True))]
    assert all(c.fast is fast for c in calls)
    for step in range(3):
        torch.cuda.synchronize()
        for buf in got.buf:
            buf.fill_(float("nan"))
        probes = [c(probe=True, flush_index=i) for i, c in enumerate(calls)]
        torch.cuda.synchronize()
        for r in range(world):
            assert torch.equal(got.buf[r].view(torch.int16), want.buf[r].view(torch.int16)), f"step {step} rank {r}"
        for i, (p, q) in enumerate(zip(probes, probes_want)):
            assert p == zc.Probe(i, q.tasks, q.reduced_elems, q.owner_tasks, q.owner_elems, q.kept_elems)
    assert zc.device_status() == 0
