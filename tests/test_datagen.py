"""The seeded input generator: its C implementation against a Python
restatement of SplitMix64 (Steele, Lea & Flood 2014), host fill against
one-by-one sampling, and the moments of the value recipes."""
import numpy as np

import datagen
from datagen import BF16, F32, NORMAL, UNIFORM, workloads

MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def mix64(z):
    z = (z + GAMMA) & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def key(seed, stream):
    return mix64(mix64(seed) ^ ((stream * 0xD1B54A32D192ED03) & MASK))


def draw(k, i):
    return mix64((k + i * GAMMA) & MASK)


def py_normal_f32(seed, stream, i, sigma):
    k = key(seed, stream)
    s = 0
    for c in range(3):
        d = draw(k, 3 * i + c)
        s += sum((d >> (16 * f)) & 0xFFFF for f in range(4))
    return np.float32(s - 393210) * np.float32(np.float32(sigma) * np.float32(2.0 ** -16))


def py_uniform_f32(seed, stream, i):
    u = (draw(key(seed, stream), i) >> 40) - 8388608
    return np.float32(u) * np.float32(2.0 ** -23)


def test_splitmix64_first_outputs():
    # SplitMix64 seeded with 0: state advances by the golden gamma, output = mix.
    # mix64 here already adds the gamma, so output k of a generator seeded with 0
    # is mix64(k * gamma).
    assert mix64(0) == 0xE220A8397B1DCDAF


def test_c_generator_matches_python_restatement():
    streams = [0, 1, 7, (3 << 16) | 2]
    idx = [0, 1, 2, 1000, 123456789]
    S = np.array([s for s in streams for _ in idx], np.uint64)
    I = np.array([i for _ in streams for i in idx], np.int64)
    got = datagen.sample_host(S, I, F32, NORMAL, seed=3, sigma=1e-3)
    want = np.array([py_normal_f32(3, int(s), int(i), 1e-3) for s, i in zip(S, I)], np.float32)
    assert np.array_equal(got, want)
    gotb = datagen.sample_host(S, I, BF16, NORMAL, seed=3, sigma=1e-3)
    assert np.array_equal(gotb, (want.view(np.uint32) >> 16).astype(np.uint16))
    gu = datagen.sample_host(S, I, F32, UNIFORM, seed=5)
    wu = np.array([py_uniform_f32(5, int(s), int(i)) for s, i in zip(S, I)], np.float32)
    assert np.array_equal(gu, wu)


def test_host_fill_equals_sampling():
    m = datagen.host_matrix(3, 5000, BF16, NORMAL, seed=9, stream0=datagen.stream_id(0, 2), col0=1234, sigma=1e-2)
    r, c = np.meshgrid(np.arange(3), np.arange(5000), indexing="ij")
    s = datagen.sample_host((2 << 16) | r.ravel(), 1234 + c.ravel(), BF16, NORMAL, seed=9, sigma=1e-2)
    assert np.array_equal(m.ravel(), s)


def test_normal_moments_and_range():
    sigma = 1e-3
    x = datagen.host_matrix(4, 250000, F32, NORMAL, seed=1, sigma=sigma).astype(np.float64)
    assert abs(x.mean()) < 0.01 * sigma
    assert abs(x.std() / sigma - 1) < 0.01
    assert np.abs(x).max() <= 6 * sigma * (1 + 1e-6)


def test_uniform_range():
    x = datagen.host_matrix(2, 200000, BF16, UNIFORM, seed=5)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert f.min() >= -1.0 and f.max() < 1.0 and abs(f.mean()) < 0.01


def test_trees_and_buckets():
    t = workloads.tree_402m()
    assert t.n_params == 243 and t.total == 402_753_536
    q = workloads.tree_qwen3_06b()
    assert q.total == 596_049_920
    L = workloads.arrival_layout(t)
    assert [b.size for b in L.buckets] == [50_350_080] + [50_348_032] * 5 + [100_663_296]
    assert sum(b.size for b in L.buckets) == t.total
    for b in L.buckets:
        assert b.size <= workloads.BUCKET_CAPACITY or len(b.tasks) == 1
        assert np.array_equal(np.cumsum(np.r_[0, b.tasks["numel"][:-1]]), b.tasks["offset"])
    tiny = workloads.tree_tiny()
    assert tiny.n_params == 16 and tiny.numel.min() >= 1 and tiny.numel.max() <= 4096


def test_straddle_tree_has_requested_straddlers():
    import oracle
    for world in (2, 4, 8, 16):
        for s in (0, 1, world - 1):
            tree = workloads.straddle_tree(world, 10000 * world + 37, s)
            om = oracle.owner_map(world, [(list(range(world)), tree.numel)])
            assert int((om["owner"] < 0).sum()) == s
