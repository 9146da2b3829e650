"""Pins of the oracle's score and calibration against things other than itself:
the explicit-RoPE definition of the logit, hand-entered frequencies, closed
forms, the pages' worked values, and algebraic identities."""
import math

import numpy as np
import pytest

import oracle as orc

RNG = np.random.default_rng(12345)


def _rand_case(n=7, d=8, n_off=5, theta=1e4, seed=0):
    rng = np.random.default_rng(seed)
    F = d // 2
    k = rng.normal(size=(n, d)) * 2.0 + 1.0
    center = rng.normal(size=(F, 2))
    c_abs = np.hypot(center[:, 0], center[:, 1])
    mean_norm = c_abs * (1.0 + rng.uniform(0.0, 1.0, size=F))
    mrl = c_abs / mean_norm
    offsets = np.array([2 ** j for j in range(n_off)], dtype=np.int64)
    return k, center, mean_norm, mrl, offsets, theta


@pytest.mark.parametrize("style", [orc.ROPE_INTERLEAVED, orc.ROPE_HALF])
@pytest.mark.parametrize("explicit_pos", [False, True])
@pytest.mark.parametrize("norm_mode", [orc.NORM_WEIGHTED, orc.NORM_UNWEIGHTED])
@pytest.mark.parametrize("theta,d", [(1e4, 8), (1e6, 16), (1.5e5, 4)])
def test_series_equals_rope_bruteforce(style, explicit_pos, norm_mode, theta, d):
    # TriAttention summary, "The attention dot product in complex form": the
    # per-band cosine series is exactly the RoPE dot product.
    k, center, m, R, offs, _ = _rand_case(n=9, d=d, seed=d + style)
    pos = RNG.integers(0, 3000, size=9) if explicit_pos else None
    p_cur = 3100
    a = orc.score_series(k, center, m, R, offs, p_cur, theta, pos=pos, style=style, norm_mode=norm_mode)
    b = orc.score_bruteforce(k, center, m, R, offs, p_cur, theta, pos=pos, style=style, norm_mode=norm_mode)
    bound = orc.score_bound(k, m, style=style)
    assert np.all(np.abs(a - b) <= 1e-9 * bound)


def _rot(x, ang):
    c, s = math.cos(ang), math.sin(ang)
    return np.array([x[0] * c - x[1] * s, x[0] * s + x[1] * c])


def test_hand_entered_frequencies_interleaved():
    # d = 4, theta = 100: omega_0 = 1, omega_1 = 100^(-2/4) = 0.1 (entered by
    # hand, not through the oracle's formula). Interleaved pairing (x0,x1),(x2,x3).
    q = np.array([0.3, -1.2, 0.7, 0.4])
    k = np.array([[1.1, 0.2, -0.5, 0.9]])
    p_q, p_k = 57 + 4, 12
    omegas = [1.0, 0.1]
    logit = 0.0
    for f, w in enumerate(omegas):
        qq = _rot(q[2 * f:2 * f + 2], w * p_q)
        kk = _rot(k[0, 2 * f:2 * f + 2], w * p_k)
        logit += qq @ kk
    center = q.reshape(2, 2)
    mean_norm = np.hypot(center[:, 0], center[:, 1])
    mrl = np.ones(2)  # R = 1 -> norm term 0
    s = orc.score_series(k, center, mean_norm, mrl, [4], 57, 100.0, pos=[p_k])
    assert s[0] == pytest.approx(logit, rel=1e-12, abs=1e-12)


def test_hand_entered_frequencies_half_split():
    # Same case with the half pairing (x0,x2),(x1,x3).
    q = np.array([0.3, -1.2, 0.7, 0.4])
    k = np.array([[1.1, 0.2, -0.5, 0.9]])
    p_q, p_k = 100 + 1, 40
    omegas = [1.0, 0.1]
    logit = 0.0
    for f, w in enumerate(omegas):
        qq = _rot(np.array([q[f], q[f + 2]]), w * p_q)
        kk = _rot(np.array([k[0, f], k[0, f + 2]]), w * p_k)
        logit += qq @ kk
    center = np.array([[q[0], q[2]], [q[1], q[3]]])
    mean_norm = np.hypot(center[:, 0], center[:, 1])
    s = orc.score_series(k, center, mean_norm, np.ones(2), [1], 100, 100.0, pos=[p_k],
                         style=orc.ROPE_HALF)
    assert s[0] == pytest.approx(logit, rel=1e-12, abs=1e-12)


def test_single_band_closed_form_signs():
    # d = 2 -> one band with omega = 1 for any theta. c = (1, 0), k = (0, 1):
    # phi = arg c - arg k = -pi/2, so S_trig = |c||k| cos(Delta + delta - pi/2)
    # = sin(Delta + delta) with Delta = p_cur - p_k. A flipped phase or a
    # flipped Delta changes the sign or the argument.
    k = np.array([[0.0, 3.0]])
    center = np.array([[1.0, 0.0]])
    R, m = 0.25, 4.0
    s = orc.score_series(k, center, [m], [R], [1], 10, 1e4, pos=[3])
    expected = 1.0 * 3.0 * math.sin(10 - 3 + 1) + (1 - R) * m * 3.0
    assert s[0] == pytest.approx(expected, rel=1e-13)


def test_offset_average_closed_form():
    # Two offsets: the score is the plain mean of the two single-offset cosines.
    k = np.array([[2.0, 0.0]])
    center = np.array([[0.0, 1.5]])  # arg c = pi/2, arg k = 0
    s = orc.score_series(k, center, [1.5], [1.0], [2, 7], 20, 1e4, pos=[5])
    expected = 0.5 * (1.5 * 2.0 * math.cos(15 + 2 + math.pi / 2) + 1.5 * 2.0 * math.cos(15 + 7 + math.pi / 2))
    assert s[0] == pytest.approx(expected, rel=1e-13, abs=1e-13)


def test_key_equals_centre_zero_distance():
    # k = c, D = {0}, p_cur = p_k, R = 1: S = sum_f |c_f|^2 = ||c||^2.
    rng = np.random.default_rng(3)
    c = rng.normal(size=(8, 2))
    k = c.reshape(1, 16)
    m = np.hypot(c[:, 0], c[:, 1])
    s = orc.score_series(k, c, m, np.ones(8), [0], 77, 1e6, pos=[77])
    assert s[0] == pytest.approx(float(np.sum(c ** 2)), rel=1e-13)


def test_norm_term_weighting():
    # S_norm = sum_f (1 - R_f) E|q_f| |k_f|; with c = 0 the trig term vanishes.
    k = np.array([[3.0, 4.0, 0.0, 2.0]])  # |k_0| = 5, |k_1| = 2
    c = np.zeros((2, 2))
    m = np.array([2.0, 10.0])
    R = np.array([0.25, 0.5])
    s_w = orc.score_series(k, c, m, R, [1, 2], 5, 1e4)
    s_u = orc.score_series(k, c, m, R, [1, 2], 5, 1e4, norm_mode=orc.NORM_UNWEIGHTED)
    assert s_w[0] == pytest.approx(0.75 * 2 * 5 + 0.5 * 10 * 2, rel=1e-14)
    assert s_u[0] == pytest.approx(2 * 5 + 10 * 2, rel=1e-14)


def test_cosine_count(golden):
    g = golden("cosine_count.json")
    F = g["bands"]
    k = np.ones((g["keys"], 2 * F))
    c = np.ones((F, 2))
    offs = [2 ** j for j in range(g["offsets"])]
    _, n_cos = orc.score_series(k, c, np.ones(F) * 2, np.full(F, 0.5), offs, 4096, 1e6,
                                return_cos_count=True)
    assert n_cos == g["cosines"]
    assert abs(n_cos - g["page_value_approx"]) / g["page_value_approx"] < 0.02


def test_calibrate_mrl_worked_example(golden):
    g = golden("mrl_three_vectors.json")
    q = np.array(g["vectors"]).reshape(1, 1, 3, 2)
    c, m, R = orc.calibrate(q, group=1)
    e = g["expected"]
    tol = g["tolerance"]
    assert c[0, 0, 0] == pytest.approx(e["center"][0], abs=tol)
    assert c[0, 0, 1] == pytest.approx(e["center"][1], abs=tol)
    assert m[0, 0] == pytest.approx(e["mean_norm"], abs=tol)
    assert R[0, 0] == pytest.approx(e["mrl"], abs=tol)
    assert 0.999 < R[0, 0] < 1.0


def test_calibrate_closed_forms():
    # Identical samples: centre = sample, R = 1 -> (1 - R) m = 0.
    q = np.tile(np.array([0.6, -0.8, 2.0, 0.0]), (1, 1, 5, 1))
    c, m, R = orc.calibrate(q, group=1)
    assert np.allclose(c[0], [[0.6, -0.8], [2.0, 0.0]], atol=1e-15)
    assert np.allclose(m[0], [1.0, 2.0], atol=1e-15)
    assert np.allclose(R[0], [1.0, 1.0], atol=1e-15)
    # Four samples symmetric about 0: c = 0, m = 1, R = 0.
    q = np.array([[1, 0], [0, 1], [-1, 0], [0, -1]], dtype=float).reshape(1, 1, 4, 2)
    c, m, R = orc.calibrate(q, group=1)
    assert np.allclose(c, 0.0, atol=1e-16) and m[0, 0] == 1.0 and R[0, 0] == 0.0


def test_calibrate_gqa_pooling_and_head_mapping():
    # Hq = 4, G = 2: KV head 0 pools query heads 0, 1; KV head 1 pools 2, 3.
    n = 3
    q = np.zeros((1, 4, n, 2))
    q[0, 0, :, :] = [1.0, 0.0]
    q[0, 1, :, :] = [-1.0, 0.0]
    q[0, 2, :, :] = [0.0, 2.0]
    q[0, 3, :, :] = [0.0, 2.0]
    c, m, R = orc.calibrate(q, group=2)
    assert np.allclose(c[0, 0], [0.0, 0.0]) and m[0, 0] == 1.0 and R[0, 0] == 0.0
    assert np.allclose(c[1, 0], [0.0, 2.0]) and m[1, 0] == 2.0 and R[1, 0] == 1.0


def test_calibrate_half_pairing():
    q = np.array([3.0, 1.0, 4.0, 0.0]).reshape(1, 1, 1, 4)
    c_i, m_i, _ = orc.calibrate(q, group=1, style=orc.ROPE_INTERLEAVED)
    c_h, m_h, _ = orc.calibrate(q, group=1, style=orc.ROPE_HALF)
    assert np.allclose(c_i[0], [[3, 1], [4, 0]]) and np.allclose(m_i[0], [math.hypot(3, 1), 4])
    assert np.allclose(c_h[0], [[3, 4], [1, 0]]) and np.allclose(m_h[0], [5, 1])


def test_norm_identity_on_calibrated_stats():
    # TriAttention summary, "Equivalent reformulation": (1 - R_f) E|q_f| = E|q_f| - |E q_f|.
    rng = np.random.default_rng(9)
    q = rng.normal(size=(2, 4, 50, 8)) + rng.normal(size=(2, 4, 1, 8)) * 3
    c, m, R = orc.calibrate(q, group=2)
    lhs = (1 - R) * m
    rhs = m - np.hypot(c[..., 0], c[..., 1])
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-13)
    assert np.all(R <= 1 + 1e-15) and np.all(R >= 0)


# ---- post-RoPE layout: RoPE of rows and its inverse -------------------------
def test_rope_rows_round_trip_and_single_band():
    rng = np.random.default_rng(21)
    for style in (0, 1):
        x = rng.normal(size=(50, 64))
        pos = rng.integers(0, 100000, size=50)
        y = orc.rope_rows(x, pos, 1e4, style=style)
        assert np.allclose(orc.rope_rows(y, pos, 1e4, style=style, inverse=True), x, atol=1e-9)
        # rotation keeps every band's magnitude
        F = 32
        def bands(v):
            return (v[:, 0::2] + 1j * v[:, 1::2]) if style == 0 else (v[:, :F] + 1j * v[:, F:])
        assert np.allclose(np.abs(bands(y)), np.abs(bands(x)), atol=1e-9)
    # d = 4, theta = 100: omega = (1, 0.1); band f multiplied by e^{i omega_f p}
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    y = orc.rope_rows(x, [7], 100.0)
    z0 = (1 + 2j) * np.exp(1j * 7.0)
    z1 = (3 + 4j) * np.exp(1j * 0.7)
    assert np.allclose(y[0], [z0.real, z0.imag, z1.real, z1.imag], atol=1e-12)


def test_post_rope_score_equals_pre_rope_score():
    rng = np.random.default_rng(22)
    n, d, F = 200, 64, 32
    k = rng.normal(size=(n, d)) + 1.5
    pos = np.sort(rng.choice(5000, size=n, replace=False))
    c = rng.normal(size=(F, 2)) * 2
    m = np.hypot(c[:, 0], c[:, 1]) * 1.3
    R = np.hypot(c[:, 0], c[:, 1]) / m
    offs = [1, 4, 16, 64]
    for style in (0, 1):
        pre = orc.score_series(k, c, m, R, offs, 5003, 1e4, pos=pos, style=style)
        kp = orc.rope_rows(k, pos, 1e4, style=style)
        post = orc.score_post_rope(kp, pos, c, m, R, offs, 5003, 1e4, style=style)
        assert np.allclose(post, pre, rtol=0, atol=1e-9 * np.abs(pre).max())
        # and the brute-force dot product of the rotated centre with the stored key
        bf = orc.score_bruteforce(k, c, m, R, offs, 5003, 1e4, pos=pos, style=style)
        assert np.allclose(post, bf, rtol=0, atol=1e-9 * np.abs(pre).max())
