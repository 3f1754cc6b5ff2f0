"""CPU pins of the oracle's alternative bound shapes (WitCert §4.3 Proposition 1; the det-tanh shape).

* two-sided: TV <= 1/2 (A/A^- - A^-/A), A^- = E_p~[e^{-c}]; the meter takes the minimum with the
  one-sided 1/2 (A^2 - 1) and 1.  Pinned by brute force (random and adversarial, float64 and 50-digit),
  by the uniform-radius closed form (where the one-sided form is the smaller), and by the page's
  massive-activation argument (one token of mass eta with a huge radius C: the one-sided form grows
  quadratically in M = eta e^C, the two-sided one linearly).
* det-tanh: TV <= tanh(max_t c_t).  Pinned by brute force and by the two-token construction that attains
  the worst case tanh(Delta / 2) of a logit perturbation bounded by Delta.
"""
import math

import mpmath as mp
import numpy as np
import pytest

from oracle import attention as A

SM = 1.0 / math.sqrt(128)


def _tv_case(rng, S, scale=1.0):
    x = rng.standard_normal(S) * 2
    c = np.abs(rng.standard_normal(S)) * scale
    eps = c * rng.choice([-1.0, 1.0], S) * rng.uniform(0, 1, S)
    return x, c, eps


@pytest.mark.parametrize("S", [1, 2, 3, 6, 30])
def test_two_sided_and_tanh_sound_brute_force(S):
    rng = np.random.default_rng(50 + S)
    for trial in range(300):
        x, c, eps = _tv_case(rng, S, scale=[0.01, 0.3, 2.0][trial % 3])
        if trial % 5 == 0:   # adversarial: every error at its bound, signs against the mass
            eps = c * np.where(np.arange(S) % 2 == 0, 1.0, -1.0)
        pt = A.softmax(x)                 # compressed distribution
        p = A.softmax(x - eps)            # exact logits x - eps
        tv = A.total_variation(p, pt)
        la = A.log_a_minus_1(np.log(pt), c)
        om = A.one_minus_a_minus(pt, c)
        assert A.two_sided_meter(la, om) >= tv - 1e-12
        assert A.det_tanh_bound(c.max()) >= tv - 1e-12
        # the unclamped two-sided form itself (Proposition 1)
        a, am = 1.0 + math.exp(la) if la > -np.inf else 1.0, 1.0 - om
        assert A.two_sided_bound(a, am) >= tv - 1e-12


def test_two_sided_mpmath_brute_force():
    mp.mp.dps = 50
    rng = np.random.default_rng(9)
    for _ in range(60):
        S = int(rng.integers(1, 5))
        x, c, eps = _tv_case(rng, S, scale=1.5)
        xs = [mp.mpf(v) for v in x]
        pt = [mp.e ** v for v in xs]
        zt = mp.fsum(pt)
        pt = [v / zt for v in pt]
        p = [mp.e ** (xs[i] - mp.mpf(eps[i])) for i in range(S)]
        z = mp.fsum(p)
        p = [v / z for v in p]
        tv = mp.fsum(abs(p[i] - pt[i]) for i in range(S)) / 2
        a = mp.fsum(pt[i] * mp.e ** mp.mpf(c[i]) for i in range(S))
        am = mp.fsum(pt[i] * mp.e ** (-mp.mpf(c[i])) for i in range(S))
        assert tv <= (a / am - am / a) / 2
        assert tv <= mp.tanh(max(mp.mpf(v) for v in c))
        # the oracle's 1 - A^- agrees with the 50-digit value
        assert abs(A.one_minus_a_minus(np.array([float(v) for v in pt]), c) - float(1 - am)) <= 1e-14


def test_uniform_radius_closed_form():
    """c_t = c for all t: A = e^c, A^- = e^{-c}; two-sided = sinh(2c) > one-sided = (e^{2c} - 1)/2."""
    for cval in (1e-4, 0.05, 0.3):
        pt = np.full(7, 1 / 7)
        c = np.full(7, cval)
        la = A.log_a_minus_1(np.log(pt), c)
        om = A.one_minus_a_minus(pt, c)
        assert om == pytest.approx(-math.expm1(-cval), rel=1e-13)
        a, am = math.exp(cval), math.exp(-cval)
        assert A.two_sided_bound(a, am) == pytest.approx(math.sinh(2 * cval), rel=1e-12)
        assert A.two_sided_meter(la, om) == pytest.approx(0.5 * math.expm1(2 * cval), rel=1e-12)


def test_massive_activation_regime():
    """One token of p~-mass eta with radius C, the rest 0: A = 1 + eta (e^C - 1), A^- = 1 - eta (1 - e^{-C})."""
    eta, C = 0.01, 10.0
    pt = np.array([eta, 1 - eta])
    c = np.array([C, 0.0])
    la = A.log_a_minus_1(np.log(pt), c)
    om = A.one_minus_a_minus(pt, c)
    a = 1 + eta * math.expm1(C)
    am = 1 - eta * (-math.expm1(-C))
    assert math.exp(la) == pytest.approx(a - 1, rel=1e-12)
    assert 1 - om == pytest.approx(am, rel=1e-12)
    M = eta * math.exp(C)
    one_sided = 0.5 * (a * a - 1)
    two_sided = A.two_sided_bound(a, am)
    assert one_sided == pytest.approx(0.5 * (M * M + 2 * M), rel=0.02)   # quadratic in M
    assert two_sided < one_sided / 50 and two_sided == pytest.approx(M / 2, rel=0.05)  # linear in M


def test_tanh_worst_case_construction():
    """Two tokens, eps = (+D, -D), p_1 = 1 / (1 + e^D): TV = tanh(D / 2) exactly, below tanh(D)."""
    for D in (0.01, 0.5, 3.0):
        a = 1 / (1 + math.exp(D))
        p = np.array([a, 1 - a])
        pt = A.softmax(np.log(p) + np.array([D, -D]))
        tv = A.total_variation(p, pt)
        assert tv == pytest.approx(math.tanh(D / 2), rel=1e-12)
        assert A.det_tanh_bound(D) >= tv


def test_decode_head_shapes_wiring():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((3, 128))
    k = rng.standard_normal((20, 128)).astype(np.float32)
    k_hat = k.astype(np.float64) + 0.05 * rng.standard_normal((20, 128))
    v = rng.standard_normal((20, 128))
    w = np.abs(rng.standard_normal((20, 16))) * 0.05
    res = A.decode_head(q, k, k_hat, v, w, SM)
    x = SM * (q @ k_hat.T)
    pt = np.exp(x - A.logsumexp(x)[:, None])
    for h in range(3):
        c = A.tier_a_radius(q[h], w, SM)
        assert res.one_minus_a_minus[h] == pytest.approx(float(pt[h] @ (1 - np.exp(-c))), rel=1e-12)
        assert res.meter_tanh[h] == pytest.approx(math.tanh(c.max()), rel=1e-14)
    assert np.all(res.meter_two_sided <= res.meter_a + 1e-15)
    assert np.all(res.meter_two_sided >= res.tv)
