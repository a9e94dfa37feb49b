"""Pins for the oracle's SAPS mask + compaction, random perfect matching,
pair averaging and the EASGD elastic step.

Sources: "Communication-Efficient Decentralized Learning with Sparsification
and Adaptive Peer Selection", section II (same mask on every worker from a
shared seed, Bernoulli(1/c); fewer than 2N/c values sent and received per
round; single-peer gossip, doubly stochastic gossip matrix).  IMerge design
notes (blog), EASGD local and global update equations.
"""
import math

import numpy as np
import pytest

import oracle

M64 = (1 << 64) - 1


def _py_uniform(key: int) -> float:
    """The counter-based uniform written independently with Python integers
    (SplitMix64, pinned by its known answers in test_oracle_qsgd)."""
    z = (key + 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    z ^= z >> 31
    return (z >> 40) / float(1 << 24)


@pytest.mark.parametrize("n,p,seed", [(1, 0.5, 3), (17, 0.3, 9), (4096, 0.01, 12345),
                                      (4096, 0.25, 2 ** 63 + 5), (1000, 1.0, 7)])
def test_mask_brute_force(n, p, seed):
    models = [np.arange(n, dtype=np.float64) * (k + 1) for k in range(3)]
    K, idx, vals = oracle.saps_mask_compact(n, p, seed, models)
    expect = [i for i in range(n) if _py_uniform(seed ^ i) < p]
    assert K == len(expect)
    assert idx.tolist() == expect
    for k in range(3):
        np.testing.assert_array_equal(vals[k], models[k][expect])


def test_mask_count_is_binomial_and_traffic_bound():
    n = 1 << 20
    for p, seed in ((0.01, 5), (0.001, 6)):
        models = [np.zeros(n)]
        K, idx, _ = oracle.saps_mask_compact(n, p, seed, models)
        pp = math.ceil(p * 2 ** 24) / 2 ** 24
        assert abs(K - n * pp) <= 5 * math.sqrt(n * pp * (1 - pp))
        c = 1 / p
        assert 2 * K < 2 * n / c + 10 * math.sqrt(n)     # traffic per worker and round
        assert np.all(np.diff(idx.astype(np.int64)) > 0)


def test_mask_same_for_every_worker_and_new_each_round():
    n = 50_000
    models = [np.random.default_rng(k).normal(size=n) for k in range(4)]
    K1, idx1, vals1 = oracle.saps_mask_compact(n, 0.01, oracle.round_seed(5, 0), models)
    K2, idx2, _ = oracle.saps_mask_compact(n, 0.01, oracle.round_seed(5, 1), models)
    for k in range(4):
        np.testing.assert_array_equal(vals1[k], models[k][idx1])
    assert not np.array_equal(idx1[:min(K1, K2)], idx2[:min(K1, K2)])


def test_capacity_truncates_but_counts_all():
    n = 10_000
    models = [np.arange(n, dtype=np.float64)]
    K, idx, vals = oracle.saps_mask_compact(n, 0.1, 77, models)
    K2, idx2, vals2 = oracle.saps_mask_compact(n, 0.1, 77, models, capacity=10)
    assert K2 == K and idx2.size == 10
    np.testing.assert_array_equal(idx2, idx[:10])


def test_round_seed_is_hash_of_base_plus_t():
    assert oracle.round_seed(0, 0) == 0xE220A8397B1DCDAF
    assert oracle.round_seed(5, 2) == oracle.splitmix64(7)


@pytest.mark.parametrize("W", [2, 4, 16, 64])
def test_matching_is_a_perfect_matching(W):
    seen = set()
    for t in range(30):
        pairs = oracle.saps_matching(oracle.round_seed(5, t), W)
        assert sorted(pairs.tolist()) == list(range(W))
        seen.add(tuple(pairs.tolist()))
        np.testing.assert_array_equal(pairs, oracle.saps_matching(oracle.round_seed(5, t), W))
    if W > 2:
        assert len(seen) > 1


def test_matching_rejects_odd_or_empty():
    for W in (0, 3, -2):
        with pytest.raises(ValueError):
            oracle.saps_matching(1, W)


def test_matching_uniform_for_four_workers():
    """Four workers have three perfect matchings; a uniform draw hits each
    about a third of the time."""
    counts = {}
    for t in range(3000):
        p = oracle.saps_matching(oracle.round_seed(11, t), 4).tolist()
        partner = {p[0]: p[1], p[1]: p[0], p[2]: p[3], p[3]: p[2]}
        counts[partner[0]] = counts.get(partner[0], 0) + 1
    assert set(counts) == {1, 2, 3}
    for c in counts.values():
        assert abs(c - 1000) < 5 * math.sqrt(3000 * (1 / 3) * (2 / 3))


def _dyadic(rng, n):
    return rng.integers(-2 ** 12, 2 ** 12, n) / 2.0 ** 8


def test_peer_average_doubly_stochastic_and_local():
    rng = np.random.default_rng(3)
    n, W = 5000, 8
    models = [_dyadic(rng, n) for _ in range(W)]
    before = [m.copy() for m in models]
    seed_t = oracle.round_seed(5, 3)
    K, idx, vals = oracle.saps_mask_compact(n, 0.05, seed_t, models)
    pairs = oracle.saps_matching(seed_t, W)
    oracle.saps_peer_average(models, vals, idx, pairs)
    # the per-coordinate sum over workers is preserved exactly
    np.testing.assert_array_equal(np.sum(models, axis=0), np.sum(before, axis=0))
    mask = np.zeros(n, bool)
    mask[idx] = True
    for q in range(W // 2):
        a, b = pairs[2 * q], pairs[2 * q + 1]
        np.testing.assert_array_equal(models[a][mask], models[b][mask])
        np.testing.assert_array_equal(models[a][mask], (before[a][mask] + before[b][mask]) / 2)
    for k in range(W):
        np.testing.assert_array_equal(models[k][~mask], before[k][~mask])


def test_easgd_special_cases():
    rng = np.random.default_rng(4)
    n, W = 300, 4
    base = [rng.normal(size=n) for _ in range(W)]
    c0 = rng.normal(size=n)
    # alpha = beta = 0: nothing moves
    m = [x.copy() for x in base]
    c = c0.copy()
    oracle.easgd_step(m, 0.0, 0.0, c)
    for x, y in zip(m, base):
        np.testing.assert_array_equal(x, y)
    np.testing.assert_array_equal(c, c0)
    # alpha = 1: every worker lands on the old center; beta = 1: center = old mean
    m = [x.copy() for x in base]
    c = c0.copy()
    oracle.easgd_step(m, 1.0, 1.0, c)
    for x in m:
        np.testing.assert_allclose(x, c0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(c, np.mean(base, axis=0), rtol=0, atol=1e-15)
    # all workers equal to the center: fixed point
    m = [c0.copy() for _ in range(W)]
    c = c0.copy()
    oracle.easgd_step(m, 0.9, 0.9, c)
    for x in m:
        np.testing.assert_array_equal(x, c0)
    np.testing.assert_allclose(c, c0, rtol=0, atol=1e-15)


def test_easgd_hand_example():
    # two workers 1 and 3, center 0, alpha 1/2, beta 1/4:
    # workers -> 1/2 and 3/2; center -> 3/4 * 0 + 1/4 * 2 = 1/2
    m = [np.array([1.0]), np.array([3.0])]
    c = np.array([0.0])
    oracle.easgd_step(m, 0.5, 0.25, c)
    assert m[0][0] == 0.5 and m[1][0] == 1.5 and c[0] == 0.5


def test_easgd_from_sum_equals_the_all_worker_step():
    """The one-worker form used when workers are separate processes: given the
    elementwise sum of the W pre-step models (summed in worker order, as the
    all-worker step sums), each worker's update and the center equal the
    all-worker EASGD step; alpha = 0 leaves the model, beta = 1 makes the
    center the mean."""
    rng = np.random.default_rng(12)
    W, n = 5, 777
    models = [rng.normal(0, 0.05, n) for _ in range(W)]
    center = rng.normal(0, 0.05, n)
    total = np.zeros(n)
    for m in models:
        total = total + m
    ref = [m.copy() for m in models]
    rc = center.copy()
    oracle.easgd_step(ref, 0.9, 0.5, rc)
    for k in range(W):
        m, c = models[k].copy(), center.copy()
        oracle.easgd_step_from_sum(m, total, W, 0.9, 0.5, c)
        np.testing.assert_array_equal(m, ref[k])
        np.testing.assert_array_equal(c, rc)
    m, c = models[0].copy(), center.copy()
    oracle.easgd_step_from_sum(m, total, W, 0.0, 1.0, c)
    np.testing.assert_array_equal(m, models[0])
    np.testing.assert_array_equal(c, total / W)
