"""The seeded input generators (no GPU): determinism, ranges, distributions."""
import numpy as np

import synth


def test_streams_are_deterministic_and_distinct():
    a = synth.u64_stream(1, 0, 1000)
    assert np.array_equal(a, synth.u64_stream(1, 0, 1000))
    assert np.array_equal(a[10:20], synth.u64_stream(1, 0, 10, start=10))
    assert not np.array_equal(a, synth.u64_stream(1, 1, 1000))
    assert not np.array_equal(a, synth.u64_stream(2, 0, 1000))
    assert len(set(a.tolist())) == 1000


def test_value_ranges_and_moments():
    u = synth.uniform_pm1_f32(2, 0, 200000)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    k = synth.int_uniform_f32(0, 0, 200000)
    assert set(np.unique(k).tolist()) == set(range(-8, 9))
    counts = np.bincount((k + 8).astype(int))
    assert counts.min() > 0.9 * counts.mean()
    z = synth.normal_f32(1, 3, 200001)
    assert z.size == 200001 and abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.mean(np.abs(z) < 1.0) > 0.67 and np.mean(np.abs(z) < 1.0) < 0.70


def test_zipf_lengths():
    R, s = 8, 0.125
    for total in (0, 1, 7, 1000, 1 << 20, (1 << 29) + 3):
        n = synth.zipf_lengths(total, R, s, seed=4)
        assert sum(n) == total and all(x >= 0 for x in n)
        w = np.array([(i + 1) ** -s for i in range(R)])
        want = sorted(total * w / w.sum())
        assert all(abs(a - b) <= 1 for a, b in zip(sorted(n), want))
    assert synth.zipf_lengths(1 << 20, R, s, 4) == synth.zipf_lengths(1 << 20, R, s, 4)
    shuffles = {tuple(synth.zipf_lengths(1 << 20, R, s, seed)) for seed in range(20)}
    assert len(shuffles) > 5
    m = synth.zipf_matrix(1 << 20, R, s, 4)
    assert all(sum(row) == 1 << 20 for row in m) and len({tuple(r) for r in m}) > 1


def test_equal_lengths():
    assert synth.equal_lengths(10, 3) == [3, 3, 4]
    assert synth.equal_lengths(4096 * 3, 3) == [4096] * 3
