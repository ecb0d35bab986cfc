"""Pins of the oracle's bucket flush (DeepSpeed issue #8700).

What pins it: PyTorch's round-to-nearest-even bf16 cast and hand-made tie
cases; the issue's exactness check (identical input on every rank reproduces
exactly); integer-valued inputs whose sums are exact; the rounding-error bound
against an exact fp64 sum; the reduce-to-owner path giving the same bits as
AllReduce on the owner ("same reduction, same operand order per element"); an
independent numpy restatement on the tiny workload; and the probe counters of
the printed probe line and the (ws-1)/ws discard rate.
"""
import numpy as np
import pytest
import torch

import oracle
from datagen import BF16, F32, NORMAL, host_matrix, workloads
from tests import np_reference as npr
from tests.helpers import holder_sets, is_sentinel, oracle_dst


# ------------------------------------------------------------------ bf16 ---

def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties
    u[:50000] = (u[:50000] & 0xFFFF0000) | 0x8000
    u[50000:60000] = (u[50000:60000] & 0xFFFF0000) | 0x7FFF
    u[60000:70000] = (u[60000:70000] & 0xFFFF0000) | 0x8001
    f = u.view(np.float32)
    got = oracle.f32_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    gotf = oracle.bf16_to_f32(got[nan])
    assert np.all(np.isnan(gotf))


def test_bf16_ties_to_even_by_hand():
    cases = {
        0x3F808000: 0x3F80,  # 1 + 2^-8: halfway between 1.0 and next, kept part even -> down
        0x3F818000: 0x3F82,  # halfway, kept part odd -> up
        0x3F808001: 0x3F81,  # just above half -> up
        0x3F807FFF: 0x3F80,  # just below half -> down
        0x7F7FFFFF: 0x7F80,  # max float rounds to +inf
        0xFF800000: 0xFF80,  # -inf stays
        0x80000000: 0x8000,  # -0 stays
        0x00000001: 0x0000,  # smallest subnormal rounds to +0
    }
    for f_bits, want in cases.items():
        f = np.array([f_bits], np.uint32).view(np.float32)
        assert int(oracle.f32_to_bf16(f)[0]) == want, hex(f_bits)


def test_bf16_widening_is_exact():
    u = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(u)
    assert np.array_equal(f.view(np.uint32), u.astype(np.uint32) << 16)


# ---------------------------------------------------- element reduction ---

@pytest.mark.parametrize("world", [2, 4, 8, 16])
def test_identical_replicas_reproduce_exactly_bf16(world):
    row = host_matrix(1, 20000, BF16, NORMAL, seed=11, sigma=1e-2)
    x = np.repeat(row, world, axis=0)
    assert np.array_equal(oracle.reduce_rows(x, pre_div=True), row[0])
    y32 = oracle.reduce_rows(x, pre_div=True, out_dt=F32)
    assert np.array_equal(y32, oracle.bf16_to_f32(row[0]))


@pytest.mark.parametrize("world", [2, 4, 8, 16])
def test_identical_replicas_reproduce_exactly_f32_short_mantissa(world):
    # values with at most 16 significant bits: k * x / W stays exact in fp32
    rng = np.random.default_rng(world)
    m = rng.integers(-(2**15), 2**15, size=5000).astype(np.float32)
    x1 = (m * np.float32(2.0 ** -20)).astype(np.float32)
    x = np.repeat(x1[None, :], world, axis=0)
    assert np.array_equal(oracle.reduce_rows(x, pre_div=True).view(np.uint32), x1.view(np.uint32))


@pytest.mark.parametrize("world", [2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("pre_div", [False, True])
def test_integer_valued_inputs_are_exact(world, pre_div):
    rng = np.random.default_rng(100 + world)
    ints = rng.integers(-128, 128, size=(world, 4000))
    x = (ints * 2.0 ** -6).astype(np.float32)
    exact = x.astype(np.float64).sum(axis=0)
    y = oracle.reduce_rows(x, pre_div=pre_div)
    if pre_div and world & (world - 1) == 0:
        assert np.array_equal(y.astype(np.float64), exact / world)
    elif not pre_div:
        assert np.array_equal(y.astype(np.float64), exact)
    # bf16 inputs with the same values (exactly representable: 8 significant bits)
    xb = npr.f32_to_bf16_bits(x)
    assert np.array_equal(oracle.bf16_to_f32(xb), x)
    yb = oracle.reduce_rows(xb, pre_div=pre_div, out_dt=F32)
    assert np.array_equal(yb, y)


@pytest.mark.parametrize("world", [2, 3, 5, 7, 8, 12, 16])
def test_rounding_error_bound_against_exact_sum(world):
    u = 2.0 ** -24
    rng = np.random.default_rng(200 + world)
    x = (rng.standard_normal((world, 20000)) * np.exp(rng.uniform(-8, 8, (world, 20000)))).astype(np.float32)
    for pre_div in (False, True):
        terms = x.astype(np.float64) / (world if pre_div else 1)
        exact = terms.sum(axis=0)
        mag = np.abs(terms).sum(axis=0)
        y = oracle.reduce_rows(x, pre_div=pre_div).astype(np.float64)
        n = world - 1
        gamma = n * u / (1 - n * u)
        bound = (gamma * (1 + u) + (u if pre_div else 0)) * mag
        assert np.all(np.abs(y - exact) <= bound * (1 + 1e-12))
        # bf16 output adds at most half an ulp of bf16 (relative 2^-8) on top
        yb = oracle.bf16_to_f32(oracle.reduce_rows(x, pre_div=pre_div, out_dt=BF16)).astype(np.float64)
        assert np.all(np.abs(yb - exact) <= bound * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y) * (1 + 1e-12))


def test_sum_starts_from_rank0_term_keeps_negative_zero():
    x = np.array([[-0.0], [-0.0]], np.float32)
    y = oracle.reduce_rows(x, pre_div=False)
    assert y.view(np.uint32)[0] == 0x80000000


# ------------------------------------------------------------ the flush ---

def _tiny(world=4, seed_grads=2):
    tree = workloads.tree_tiny(seed=1)
    layout = workloads.arrival_layout(tree, capacity=None)
    assert len(layout.buckets) == 1
    b = layout.buckets[0]
    grads = host_matrix(world, b.size, BF16, NORMAL, seed=seed_grads, sigma=1e-2)
    return tree, b, grads


@pytest.mark.parametrize("reduce_to_owner", [True, False])
@pytest.mark.parametrize("out_bf16", [True, False])
def test_tiny_flush_matches_independent_numpy(reduce_to_owner, out_bf16):
    world = 4
    tree, b, grads = _tiny(world)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)], reduce_to_owner)
    holders = holder_sets(om["holder_lo"], om["holder_hi"])
    assert any(len(h) > 1 for h in holders), "the tiny workload must contain straddlers"
    dst = oracle_dst(world, b.tasks, holders, out_bf16)
    probe = oracle.flush(world, grads.copy(), b.tasks, om["owner"], tree.n_params, dst, BF16 if out_bf16 else F32,
                         pre_div=True, reduce_to_owner=reduce_to_owner)
    ref = npr.flush(world, npr.bf16_bits_to_f32(grads), b.tasks, om["owner"], reduce_to_owner, True, out_bf16,
                    holders)
    for t, task in enumerate(b.tasks):
        pid = int(task["param_id"])
        for r in range(world):
            if dst[r][t] is None:
                continue
            if (r, pid) in ref:
                want = ref[(r, pid)]
                assert np.array_equal(dst[r][t].view(want.dtype), want), (r, pid)
            else:
                assert np.all(is_sentinel(dst[r][t], out_bf16)), "non-delivered buffer was written"
    assert probe["tasks"] == len(b.tasks) and probe["reduced_elems"] == b.size


def test_rank_order_matters_vacuity_guard():
    """A different summation order gives different bits on this data, so the
    bit-exact comparisons above can fail."""
    world = 8
    x = npr.bf16_bits_to_f32(host_matrix(world, 50000, BF16, NORMAL, seed=5, sigma=1e-2))
    fwd = npr.reduce_f32(x, True)
    rev = npr.reduce_f32(x, True, order=range(world - 1, -1, -1))
    assert not np.array_equal(fwd, rev)
    assert np.array_equal(oracle.reduce_rows(x, pre_div=True), fwd)


def test_owner_path_gives_allreduce_bits_on_owner():
    world = 4
    tree, b, grads = _tiny(world)
    on = oracle.owner_map(world, [(list(range(world)), tree.numel)], True)
    holders = holder_sets(on["holder_lo"], on["holder_hi"])
    d_owner = oracle_dst(world, b.tasks, holders, True)
    d_ar = oracle_dst(world, b.tasks, holders, True)
    oracle.flush(world, grads.copy(), b.tasks, on["owner"], tree.n_params, d_owner, BF16, True, True)
    oracle.flush(world, grads.copy(), b.tasks, on["owner"], tree.n_params, d_ar, BF16, True, False)
    for t in range(len(b.tasks)):
        for r in range(world):
            if d_owner[r][t] is not None:
                # holders only ever have the owner (owner tasks) or all holders (straddlers) delivered
                assert np.array_equal(d_owner[r][t], d_ar[r][t])


def test_in_place_owner_writes_only_owner_row():
    world = 4
    tree, b, grads = _tiny(world)
    on = oracle.owner_map(world, [(list(range(world)), tree.numel)], True)
    before = grads.copy()
    g = grads.copy()
    probe = oracle.flush(world, g, b.tasks, on["owner"], tree.n_params, None, BF16, True, True)
    ar = before.copy()
    oracle.flush(world, ar, b.tasks, on["owner"], tree.n_params, None, BF16, True, False)
    for task in b.tasks:
        pid, off, n = int(task["param_id"]), int(task["offset"]), int(task["numel"])
        own = on["owner"][pid]
        want = oracle.reduce_rows(before[:, off:off + n], pre_div=True)
        for r in range(world):
            seg = g[r, off:off + n]
            if own < 0 or own == r:
                assert np.array_equal(seg, want)
            else:
                assert np.array_equal(seg, before[r, off:off + n])
            assert np.array_equal(ar[r, off:off + n], want)
    straddle = sum(int(t["numel"]) for t in b.tasks if on["owner"][int(t["param_id"])] < 0)
    assert probe["owner_elems"] == b.size - straddle


# -------------------------------------------------------------- probe ---

def _partitioned_bucket(world, per_rank_sizes):
    """A group made of whole-partition parameters: rank j's partition holds the
    parameters listed in per_rank_sizes[j] (all partitions the same size)."""
    sizes = [s for part in per_rank_sizes for s in part]
    tree = workloads.Tree([f"p{i}" for i in range(len(sizes))], np.array(sizes, np.int64))
    return tree, workloads.arrival_layout(tree, capacity=None).buckets[0]


def test_probe_reproduces_printed_line_counters(golden_dir):
    """The bucket of the printed probe line: W=8, 118 tasks, 52,428,800 elements,
    rank 0 keeping 6,553,600, flag off."""
    world = 8
    per = 52_428_800 // world
    per_rank = []
    for j in range(world):
        k = 15 if j < 6 else 14           # 6*15 + 2*14 = 118 tasks
        base = per // k
        sizes = [base] * (k - 1) + [per - base * (k - 1)]
        per_rank.append(sizes)
    tree, b = _partitioned_bucket(world, per_rank)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)], reduce_to_owner=False)
    has = np.zeros((world, len(b.tasks)), bool)
    for t, task in enumerate(b.tasks):
        p = int(task["param_id"])
        has[om["holder_lo"][p]:om["holder_hi"][p] + 1, t] = True
    pr = oracle.flush_probe(world, b.tasks, om["owner"], tree.n_params, has, reduce_to_owner=False)
    fields = {}
    for line in open(f"{golden_dir}/probe_line.txt"):
        if line.startswith("[dc-probe]"):
            for tok in line.split():
                if "=" in tok:
                    k, v = tok.split("=", 1)
                    fields[k] = v
    assert pr["tasks"] == int(fields["tasks"]) == 118
    assert pr["reduced_elems"] == int(fields["reduced_elems"])
    assert pr["kept_elems"][0] == int(fields["kept_elems"])
    discarded = 100.0 * (pr["reduced_elems"] - pr["kept_elems"][0]) / pr["reduced_elems"]
    assert f"{discarded:.1f}%" == fields["discarded"]
    assert pr["owner_tasks"] == int(fields["owner_tasks"]) and pr["owner_elems"] == int(fields["owner_elems"])
    # with the flag on every task of this bucket takes the owner path
    om_on = oracle.owner_map(world, [(list(range(world)), tree.numel)], reduce_to_owner=True)
    pr_on = oracle.flush_probe(world, b.tasks, om_on["owner"], tree.n_params, has, reduce_to_owner=True)
    assert pr_on["owner_tasks"] == 118 and pr_on["owner_elems"] == 52_428_800
    assert pr_on["kept_elems"] == pr["kept_elems"]


@pytest.mark.parametrize("world", [2, 4, 8, 16])
def test_discarded_fraction_is_ws_minus_one_over_ws(world):
    per_rank = [[1000 + 37 * j, 2000, 513] for j in range(world)]
    per_rank = [[s for s in part] for part in per_rank]
    # equalise partitions so that no parameter straddles
    tot = max(sum(p) for p in per_rank)
    per_rank = [p[:-1] + [p[-1] + tot - sum(p)] for p in per_rank]
    tree, b = _partitioned_bucket(world, per_rank)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)])
    assert np.all(om["owner"] >= 0)
    has = np.zeros((world, len(b.tasks)), bool)
    for t, task in enumerate(b.tasks):
        p = int(task["param_id"])
        has[om["holder_lo"][p]:om["holder_hi"][p] + 1, t] = True
    pr = oracle.flush_probe(world, b.tasks, om["owner"], tree.n_params, has, reduce_to_owner=False)
    assert sum(pr["kept_elems"]) == pr["reduced_elems"]
    mean_discard = np.mean([(pr["reduced_elems"] - k) / pr["reduced_elems"] for k in pr["kept_elems"]])
    assert abs(mean_discard - (world - 1) / world) < 1e-12


def test_probe_owner_elems_excludes_straddlers():
    tree = workloads.tree_402m()
    om = oracle.owner_map(8, [(list(range(8)), tree.numel)], True)
    layout = workloads.arrival_layout(tree)
    total_owner = 0
    for b in layout.buckets:
        pr = oracle.flush_probe(8, b.tasks, om["owner"], tree.n_params, None, True)
        strad = sum(int(t["numel"]) for t in b.tasks if om["owner"][int(t["param_id"])] < 0)
        assert pr["owner_elems"] == pr["reduced_elems"] - strad
        total_owner += pr["owner_elems"]
    assert total_owner == 295_798_784


def test_wrong_root_is_caught_vacuity_guard():
    """A plausible mistake -- every owner shifted to the next rank -- changes
    both the delivered buffers and the kept counts, so the parity checks that
    compare them would fail on it."""
    world = 4
    tree, b, grads = _tiny(world)
    om = oracle.owner_map(world, [(list(range(world)), tree.numel)], True)
    holders = holder_sets(om["holder_lo"], om["holder_hi"])
    right = oracle_dst(world, b.tasks, holders, True)
    wrong = oracle_dst(world, b.tasks, holders, True)
    bad_owner = np.where(om["owner"] >= 0, (om["owner"] + 1) % world, -1).astype(np.int32)
    pr_right = oracle.flush(world, grads.copy(), b.tasks, om["owner"], tree.n_params, right, BF16, True, True)
    oracle.flush(world, grads.copy(), b.tasks, bad_owner, tree.n_params, wrong, BF16, True, True)
    differs = any(not np.array_equal(right[r][t], wrong[r][t])
                  for r in range(world) for t in range(len(b.tasks)) if right[r][t] is not None)
    assert differs
    has = np.array([[right[r][t] is not None for t in range(len(b.tasks))] for r in range(world)])
    assert oracle.flush_probe(world, b.tasks, bad_owner, tree.n_params, None, True)["kept_elems"] != \
        oracle.flush_probe(world, b.tasks, om["owner"], tree.n_params, None, True)["kept_elems"]
    assert pr_right["kept_elems"] == oracle.flush_probe(world, b.tasks, om["owner"], tree.n_params, has, True)["kept_elems"]
