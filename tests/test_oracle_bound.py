"""Pins of oracle.score_bound, the scale M(i) = sum_f E|q_f| |k_f| of every
score tolerance in the GPU parity tests.

Why M bounds the score (TriAttention summary page, section 3.4, "The
Norm-Based Term" and "Adaptive Weighting via Q/K Concentration"): the
trigonometric term of band f is at most |E q_f| |k_f| in magnitude (the
offset average G_f has modulus <= 1), the weighted norm term adds
(E|q_f| - |E q_f|) |k_f| >= 0, and |E q_f| <= E|q_f| (the modulus of a mean is
at most the mean modulus). So |S~(i)| <= M(i), with equality when the
statistics are concentrated (R_f = 1) and every band's phase lines up, and
S~(i) = M(i) exactly when the query centre is zero. With the unweighted norm
term (E|q_f| |k_f| in full) the score lies in [0, 2 M(i)].

The hand-entered values below are computed on paper, not through the
oracle, so a dropped square root, a squared mean norm or a wrong band
pairing in score_bound fails them.
"""
import math

import numpy as np
import pytest

import oracle as orc


def test_hand_entered_bound_interleaved():
    # d = 4, interleaved bands (k0, k1) = (3, 4) and (k2, k3) = (1, 0):
    # |k_0| = 5, |k_1| = 1; E|q| = (2, 0.5) -> M = 2*5 + 0.5*1 = 10.5.
    k = np.array([[3.0, 4.0, 1.0, 0.0]])
    m = np.array([2.0, 0.5])
    assert orc.score_bound(k, m, style=orc.ROPE_INTERLEAVED)[0] == pytest.approx(10.5, rel=1e-15)


def test_hand_entered_bound_half_split():
    # Same key, half pairing: bands (k0, k2) = (3, 1) and (k1, k3) = (4, 0):
    # |k_0| = sqrt(10), |k_1| = 4 -> M = 2*sqrt(10) + 0.5*4.
    k = np.array([[3.0, 4.0, 1.0, 0.0]])
    m = np.array([2.0, 0.5])
    want = 2.0 * math.sqrt(10.0) + 2.0
    assert orc.score_bound(k, m, style=orc.ROPE_HALF)[0] == pytest.approx(want, rel=1e-15)


def test_hand_entered_bound_several_rows():
    # Rows are independent and the bound is linear in E|q_f|.
    k = np.array([[3.0, 4.0, 1.0, 0.0], [0.0, 0.0, 0.0, 0.0], [-6.0, 8.0, 0.0, -2.0]])
    m = np.array([1.0, 3.0])
    got = orc.score_bound(k, m)
    assert got == pytest.approx([5.0 + 3.0, 0.0, 10.0 + 6.0], rel=1e-15)
    assert orc.score_bound(k, 2.0 * m) == pytest.approx(2.0 * got, rel=1e-15)


def _calibrated_case(seed, d, style, n_q=64, spread=1.0):
    """Statistics from real calibration (so E|q_f| >= |E q_f| holds as it does
    in use), keys with a mean and noise, explicit positions."""
    rng = np.random.default_rng(seed)
    mu = rng.normal(size=d) * 2.0
    q = (mu + spread * rng.normal(size=(n_q, d)))[None, None]
    center, mean_norm, mrl = orc.calibrate(q, group=1, style=style)
    k = rng.normal(size=(40, d)) * rng.uniform(0.2, 3.0) + rng.normal(size=d)
    pos = rng.integers(0, 5000, size=40)
    return k, center[0], mean_norm[0], mrl[0], pos


@pytest.mark.parametrize("style", [orc.ROPE_INTERLEAVED, orc.ROPE_HALF])
@pytest.mark.parametrize("d", [4, 16, 64])
@pytest.mark.parametrize("seed", range(4))
def test_score_within_bound(style, d, seed):
    k, c, m, R, pos = _calibrated_case(seed * 7 + d, d, style, spread=0.3 + seed)
    offs = [1, 2, 4, 8, 16, 32]
    M = orc.score_bound(k, m, style=style)
    s = orc.score_series(k, c, m, R, offs, 5100, 1e4, pos=pos, style=style, norm_mode=orc.NORM_WEIGHTED)
    assert np.all(np.abs(s) <= M * (1 + 1e-12))
    s0 = orc.score_series(k, c, m, R, offs, 5100, 1e4, pos=pos, style=style, norm_mode=orc.NORM_UNWEIGHTED)
    assert np.all(s0 >= -1e-12 * M) and np.all(s0 <= 2.0 * M * (1 + 1e-12))


@pytest.mark.parametrize("style", [orc.ROPE_INTERLEAVED, orc.ROPE_HALF])
def test_zero_centre_attains_bound(style):
    # Symmetric calibration samples (q and -q) give E q_f = 0, R_f = 0: the
    # trigonometric term vanishes and the weighted norm term is M itself.
    rng = np.random.default_rng(3)
    d = 8
    half = rng.normal(size=(32, d))
    q = np.concatenate([half, -half])[None, None]
    c, m, R = (a[0] for a in orc.calibrate(q, group=1, style=style))
    assert np.all(np.abs(c) < 1e-12)
    k = rng.normal(size=(10, d)) * 3.0
    M = orc.score_bound(k, m, style=style)
    for mode in (orc.NORM_WEIGHTED, orc.NORM_UNWEIGHTED):
        s = orc.score_series(k, c, m, R, [1, 4, 16], 300, 1e4, style=style, norm_mode=mode)
        assert s == pytest.approx(M, rel=1e-12)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_aligned_single_band_attains_bound(sign):
    # One band (d = 2), concentrated statistics (E|q| = |E q|, R = 1, no norm
    # term), k = +-c, one offset 0 and the query at the key's own position:
    # S = +-|c|^2 = +-M.
    c = np.array([[1.5, -2.0]])
    m = np.array([2.5])
    k = sign * c.copy()
    M = orc.score_bound(k, m)
    assert M[0] == pytest.approx(6.25, rel=1e-15)
    s = orc.score_series(k, c, m, np.ones(1), [0], 77, 1e4, pos=[77])
    assert s[0] == pytest.approx(sign * 6.25, rel=1e-12)


def test_bound_is_tight_over_phases():
    # With R = 1 and one band, S/M = cos(angle between the rotated centre and
    # the key): over many ages its maximum approaches 1 and its minimum -1.
    c = np.array([[0.6, 0.8]])
    m = np.array([1.0])
    k = np.array([[2.0, 0.0]])
    pos = np.arange(0, 4000)
    kk = np.repeat(k, len(pos), axis=0)
    s = orc.score_series(kk, c, m, np.ones(1), [0], 4000, 10.0, pos=pos)
    M = orc.score_bound(kk, m)
    r = s / M
    assert r.max() > 0.9999 and r.min() < -0.9999 and np.all(np.abs(r) <= 1 + 1e-12)
