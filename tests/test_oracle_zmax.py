"""Pins of the oracle's GQA aggregation (TriAttention summary page,
"Handling Grouped-Query Attention"): per-head z-score over all cached keys,
then the maximum over the heads that share a KV head."""
import math

import numpy as np

import oracle as orc


def test_two_head_example_in_closed_form():
    # head 0 = 1, 2, 3, 4: mean 5/2, variance 5/4; head 1 = 10, 0, 0, 0:
    # mean 5/2, variance 75/4
    mean, std, final = orc.zscore_max([[1, 2, 3, 4], [10, 0, 0, 0]])
    assert np.allclose(mean, [2.5, 2.5], rtol=0, atol=1e-15)
    assert np.allclose(std, [math.sqrt(5) / 2, math.sqrt(75) / 2], rtol=1e-15)
    r5 = math.sqrt(5)
    # key 0: head 1 wins with 7.5 / (sqrt(75)/2) = sqrt(3); keys 1-3: head 0
    assert np.allclose(final, [math.sqrt(3), -1 / r5, 1 / r5, 3 / r5], rtol=1e-14)


def test_positive_affine_map_of_a_head_changes_nothing():
    rng = np.random.default_rng(0)
    s = rng.normal(size=(4, 500)) * [[1], [10], [0.1], [3]] + [[0], [-5], [100], [2]]
    _, _, f0 = orc.zscore_max(s)
    t = s * np.array([[2.0], [0.5], [7.0], [1.0]]) + np.array([[3.0], [-1.0], [0.0], [-9.0]])
    _, _, f1 = orc.zscore_max(t)
    assert np.allclose(f0, f1, rtol=0, atol=1e-10)


def test_single_head_is_its_z_score_with_unit_variance():
    rng = np.random.default_rng(1)
    s = rng.gamma(2.0, size=(1, 777)) * 4 - 3
    mean, std, final = orc.zscore_max(s)
    assert abs(final.mean()) < 1e-12
    assert abs(np.sqrt(np.mean(final ** 2)) - 1.0) < 1e-12  # population variance 1
    # the ordering is the raw score's, so the selection is the same
    assert np.array_equal(orc.select(final, 777, 10, 20, 200), orc.select(s[0], 777, 10, 20, 200))


def test_constant_head_contributes_zero():
    rng = np.random.default_rng(2)
    s = np.vstack([np.full(300, 4.25), rng.normal(size=300)])
    mean, std, final = orc.zscore_max(s)
    assert std[0] == 0.0 and mean[0] == 4.25
    z1 = (s[1] - s[1].mean()) / s[1].std()
    assert np.allclose(final, np.maximum(z1, 0.0), rtol=0, atol=1e-12)
    _, _, fc = orc.zscore_max(np.full((3, 50), -1.0))
    assert np.all(fc == 0.0)


def test_final_is_the_largest_head_z_score():
    rng = np.random.default_rng(3)
    s = rng.normal(size=(3, 400)) * [[1], [2], [5]]
    mean, std, final = orc.zscore_max(s)
    z = (s - mean[:, None]) / std[:, None]
    assert np.all(final >= z.max(axis=0) - 1e-12) and np.all(final <= z.max(axis=0) + 1e-12)
    assert np.all(np.isclose(z, final[None, :], rtol=0, atol=1e-12).any(axis=0))


def test_identical_heads_reduce_to_the_pooled_score():
    rng = np.random.default_rng(4)
    n, d, F = 300, 64, 32
    k = rng.normal(size=(n, d)) + 2.0
    c = rng.normal(size=(F, 2)) * 3
    m = np.hypot(c[:, 0], c[:, 1]) * 1.2
    R = np.hypot(c[:, 0], c[:, 1]) / m
    offs = [1, 2, 4, 8]
    pooled = orc.score_series(k, c, m, R, offs, n - 1, 1e4)
    heads = orc.score_heads(k, np.stack([c, c]), np.stack([m, m]), np.stack([R, R]), offs, n - 1, 1e4)
    assert np.array_equal(heads[0], pooled) and np.array_equal(heads[1], pooled)
    _, _, final = orc.zscore_max(heads)
    assert np.array_equal(orc.select(final, n, 8, 16, 100), orc.select(pooled, n, 8, 16, 100))
