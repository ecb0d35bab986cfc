"""Pins of the oracle's deferred accumulation (MaxText PR #5099, "What" and
"Results": the cross-replica addition moves from before the micro-batch sum to
after it; exact where the reassociation is exact, within 4.5e-5 relative
otherwise).  Checked against exact integer sums, the single-micro-batch case,
an exact fp64 sum with its error bound, and the per-micro-batch path."""
import numpy as np
import pytest

import oracle
from datagen import BF16, F32, NORMAL, host_matrix, stream_id


def _grads(world, n_mb, n, dt=F32, seed=4, sigma=1e-3):
    return np.stack([host_matrix(world, n, dt, NORMAL, seed=seed, stream0=stream_id(0, m), sigma=sigma)
                     for m in range(n_mb)])


def _deferred(g, scale=1.0):
    M, W, n = g.shape
    acc = np.full((W, n), np.nan, np.float32)  # garbage: `first` must overwrite it
    for m in range(M - 1):
        oracle.accumulate(acc, g[m], first=(m == 0), finalize=False)
    before = acc.copy()
    total = oracle.accumulate(acc, g[M - 1], first=(M == 1), finalize=True, scale=scale)
    assert np.array_equal(acc, before, equal_nan=True), "finalize must leave the accumulator unchanged"
    return total


@pytest.mark.parametrize("world", [1, 2, 4])
def test_single_microbatch_deferred_equals_per_microbatch(world):
    g = _grads(world, 1, 3000)
    assert np.array_equal(_deferred(g), oracle.reduce_each_microbatch(g))


@pytest.mark.parametrize("world,n_mb", [(2, 3), (4, 8), (8, 4), (3, 5)])
def test_integer_valued_inputs_agree_exactly(world, n_mb):
    rng = np.random.default_rng(world * 10 + n_mb)
    g = (rng.integers(-1000, 1000, size=(n_mb, world, 2000)) * 2.0 ** -10).astype(np.float32)
    exact = g.astype(np.float64).sum(axis=(0, 1))
    d = _deferred(g)
    p = oracle.reduce_each_microbatch(g)
    assert np.array_equal(d.astype(np.float64), exact) and np.array_equal(p.astype(np.float64), exact)


@pytest.mark.parametrize("world,n_mb", [(4, 8), (2, 4), (8, 2)])
def test_general_inputs_within_reassociation_tolerance(world, n_mb):
    g = _grads(world, n_mb, 20000)
    d = _deferred(g).astype(np.float64)
    p = oracle.reduce_each_microbatch(g).astype(np.float64)
    exact = g.astype(np.float64).sum(axis=(0, 1))
    mag = np.abs(g.astype(np.float64)).sum(axis=(0, 1))
    assert np.linalg.norm(d - p) / np.linalg.norm(p) <= 5e-5
    assert np.all(np.abs(d - p) <= 5e-5 * mag)
    # each is within the recursive-summation bound of the exact sum
    k = world * n_mb - 1
    gamma = k * 2.0 ** -24 / (1 - k * 2.0 ** -24)
    assert np.all(np.abs(d - exact) <= gamma * mag * (1 + 1e-12))
    assert np.all(np.abs(p - exact) <= gamma * mag * (1 + 1e-12))
    # the two orders really differ on this data (the comparison has teeth)
    assert not np.array_equal(d, p)


def test_world_one_finalize_is_the_accumulator():
    g = _grads(1, 3, 5000)
    acc = np.empty((1, 5000), np.float32)
    oracle.accumulate(acc, g[0], True, False)
    oracle.accumulate(acc, g[1], False, False)
    want = (acc[0] + g[2][0]).astype(np.float32)
    total = oracle.accumulate(acc, g[2], False, True)
    assert np.array_equal(total, want)


def test_first_overwrites_and_bf16_gradients_widen_exactly():
    g = _grads(4, 1, 4000, dt=BF16)[0]
    acc = np.full((4, 4000), 123.0, np.float32)
    oracle.accumulate(acc, g, first=True, finalize=False)
    assert np.array_equal(acc, oracle.bf16_to_f32(g))
    oracle.accumulate(acc, g, first=False, finalize=False)
    assert np.array_equal(acc, 2 * oracle.bf16_to_f32(g))


def test_scale_is_applied_after_the_sum():
    g = _grads(4, 2, 3000)
    plain = _deferred(g, 1.0)
    quarter = _deferred(g, 0.25)
    assert np.array_equal(quarter, (plain * np.float32(0.25)).astype(np.float32))
    third = _deferred(g, np.float32(1 / 3))
    assert np.array_equal(third, (plain * np.float32(1 / 3)).astype(np.float32))


def test_restore_form_reproduces_total():
    """A reduced total placed on replica 0 with zeros elsewhere is reproduced
    exactly by the deferred reduction (PR #5099, "Accumulator lifetime")."""
    g = _grads(4, 3, 3000)
    total = _deferred(g)
    acc = np.zeros((4, 3000), np.float32)
    acc[0] = total
    zeros = np.zeros((4, 3000), np.float32)
    out = oracle.accumulate(acc, zeros, first=False, finalize=True)
    assert np.array_equal(out, total)


def test_checkpoint_restore_then_save_reproduces_total():
    """PR #5099, "Accumulator lifetime": both directions are exact -- restoring
    a total onto one replica with zeros elsewhere and reducing again gives the
    total back (bit for bit, except that -0 becomes +0 once a +0 is added)."""
    g = _grads(4, 3, 5000)
    total = _deferred(g)
    acc = oracle.accumulator_restore(total, 4)
    assert np.array_equal(acc[0], total) and not acc[1:].any()
    again = oracle.accumulator_save(acc)
    assert np.array_equal(again.view(np.uint32), (total + np.float32(0)).view(np.uint32))


def test_save_equals_finalize_with_zero_gradient():
    g = _grads(4, 2, 4000)
    acc = np.empty((4, 4000), np.float32)
    oracle.accumulate(acc, g[0], True, False)
    oracle.accumulate(acc, g[1], False, False)
    saved = oracle.accumulator_save(acc)
    fin = oracle.accumulate(acc.copy(), np.zeros_like(acc), False, True)
    assert np.array_equal(saved, fin)   # x + 0 == x for every finite nonzero x, and the sums match
    assert np.array_equal(saved, oracle.reduce_each_microbatch(acc[None]))


@pytest.mark.parametrize("world,n_mb,cut", [(4, 8, 3), (2, 5, 1), (8, 4, 2)])
def test_mid_step_round_trip_matches_uninterrupted_run(world, n_mb, cut):
    """The mid-step checkpoint round trip of PR #5099's tests: exact on
    integer-valued gradients (reassociation is exact there), within the
    reassociation tolerance otherwise."""
    rng = np.random.default_rng(world + n_mb)
    gi = (rng.integers(-500, 500, size=(n_mb, world, 3000)) * 2.0 ** -9).astype(np.float32)
    for g, exact in ((gi, True), (_grads(world, n_mb, 3000), False)):
        straight = _deferred(g)
        acc = np.empty((world, g.shape[2]), np.float32)
        for m in range(cut):
            oracle.accumulate(acc, g[m], m == 0, False)
        acc = oracle.accumulator_restore(oracle.accumulator_save(acc), world)   # save, then restore
        for m in range(cut, n_mb - 1):
            oracle.accumulate(acc, g[m], False, False)
        resumed = oracle.accumulate(acc, g[n_mb - 1], False, True)
        if exact:
            assert np.array_equal(resumed, straight)
        else:
            d, s = resumed.astype(np.float64), straight.astype(np.float64)
            assert np.linalg.norm(d - s) / np.linalg.norm(s) <= 5e-5
