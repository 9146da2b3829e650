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


# ---- union-based selection across heads --------------------------------------
def _brute_union(s, n, P, W, B, k):
    """Direct set construction: each head's top-k candidates (stable by slot),
    their union ranked by the z-score maximum, then the rest by it."""
    H = s.shape[0]
    cand = list(range(P, n - W))
    _, _, comb = orc.zscore_max(s)
    union = set()
    for h in range(H):
        ranked = sorted(cand, key=lambda i: (-s[h, i], i))
        union |= set(ranked[:k])
    need = B - P - W
    in_u = sorted(union, key=lambda i: (-comb[i], i))
    rest = sorted(set(cand) - union, key=lambda i: (-comb[i], i))
    chosen = (in_u + rest)[:need]
    return sorted(list(range(P)) + chosen + list(range(n - W, n)))


def test_union_select_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(20):
        H, n = int(rng.integers(1, 5)), int(rng.integers(20, 80))
        s = np.round(rng.normal(size=(H, n)) * 3) / 3 * rng.uniform(0.5, 5, size=(H, 1))  # ties, scales
        P, W = int(rng.integers(0, 5)), int(rng.integers(0, 5))
        B = int(rng.integers(P + W + 1, n))
        k = int(rng.integers(0, n))
        keep, member, comb = orc.union_select(s, n, P, W, B, k)
        assert keep.tolist() == _brute_union(s, n, P, W, B, k), trial
        assert member.sum() <= H * k


def test_union_select_reductions():
    rng = np.random.default_rng(6)
    s = rng.normal(size=(4, 300)) * [[1], [3], [0.5], [2]]
    n, P, W, B = 300, 10, 20, 100
    need = B - P - W
    _, _, comb = orc.zscore_max(s)
    top = orc.select(comb, n, P, W, B)
    # every head keeps >= need of its own: the union holds the top by the maximum
    assert np.array_equal(orc.union_select(s, n, P, W, B, need)[0], top)
    # an empty union: filled by the combined score alone
    assert np.array_equal(orc.union_select(s, n, P, W, B, 0)[0], top)
    # one head: the plain selection on its score, whatever k
    for k in (0, 5, need, 200):
        assert np.array_equal(orc.union_select(s[1:2], n, P, W, B, k)[0], orc.select(s[1], n, P, W, B))
    # a small k changes the result: union members beat higher combined scores
    keep_small = orc.union_select(s, n, P, W, B, 3)[0]
    assert len(set(keep_small.tolist())) == B
    # nothing to evict
    assert orc.union_select(s[:, :90], 90, P, W, B, 3)[0].tolist() == list(range(90)) + [-1] * 10


def test_shared_draw_is_one_keep_set_for_every_head():
    a = [orc.rand_select_shared(3, 1, 0, 2, h, 1, 900, 50, 0, 300) for h in range(4)]
    assert all(np.array_equal(a[0], x) for x in a)
    assert np.array_equal(a[0], orc.rand_select(3, 1, 0, 2, 0, 900, 50, 0, 300))
    b = orc.rand_select_shared(3, 1, 0, 2, 3, 2, 900, 50, 0, 300)
    assert np.array_equal(b, orc.rand_select(3, 1, 0, 0, 0, 900, 50, 0, 300))
    assert np.array_equal(orc.rand_select_shared(3, 1, 0, 2, 3, 0, 900, 50, 0, 300),
                          orc.rand_select(3, 1, 0, 2, 3, 900, 50, 0, 300))


def test_union_steps_compose():
    rng = np.random.default_rng(7)
    s = rng.normal(size=(3, 200)) * [[1], [4], [2]]
    keep, member, comb = orc.union_select(s, 200, 5, 7, 80, 10)
    assert np.array_equal(orc.union_members(s, 5, 7, 10), member)
    assert np.array_equal(orc.union_rank(member, comb, 5, 7, 80), keep)
