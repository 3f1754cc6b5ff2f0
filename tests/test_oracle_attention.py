"""Pins of the oracle's attention, total variation and meter (CPU).

* Golden two-token counterexample printed in WitCert §3 (TV 0.049834, flawed
  Eq. (1) 0.006423) and Theorem 1's bound on it.
* Brute force at 50 digits (mpmath) on S <= 8: output, TV, ln(A - 1), Tier B.
* Adversarial Theorem 1 trials (sign patterns, peaked / flat p~, large c),
  asserted per trial, never in aggregate (WitCert §3 methodological lesson).
* Theorem 2: |eps_t| <= c_t per token; equality when q_b is parallel to r_b.
* Identity quantizer: bound 0 and TV 0.
* Joint RoPE shift of keys and query leaves TV, c_t and the bound unchanged.
* Lemma 2 closed form; Tier B zero violations over dither seeds.
* Proposition 1 example (A = 2, A^- = 0.6).
* Split-KV merge of ln(A - 1) under LSE weights equals the unsplit value.
"""
import json
import math
import os

import mpmath as mp
import numpy as np
import pytest

from oracle import attention as A
from oracle.encoders import fp16_value
from oracle.philox import dither
from oracle.quant import dequantize, quantize, witness_bits
from workloads import rope_tables

GOLD = os.path.join(os.path.dirname(__file__), "golden")
SM = 1.0 / math.sqrt(128)


def _golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_two_token_counterexample_golden():
    g = _golden("two_token_counterexample.json")
    pt = np.array(g["p_tilde"])
    c = np.array(g["c"])
    eps = np.array(g["eps"])
    # p_t is proportional to p~_t e^{-eps_t} (eps = compressed - exact logit)
    p = pt * np.exp(-eps)
    p /= p.sum()
    tv = float(A.total_variation(p, pt))
    assert round(tv, g["printed_digits"]) == g["true_tv_printed"]
    flawed = A.flawed_dispersion_bound(pt, c)
    assert round(flawed, g["printed_digits"]) == g["flawed_eq1_printed"]
    assert round(tv / flawed, 1) == g["printed_ratio"]
    # Theorem 1 on the same case: 1/2 (e^{0.2} - 1) >= TV
    lam1 = A.log_a_minus_1(np.log(pt), c)
    meter = float(A.meter_from_log_am1(lam1))
    assert meter == pytest.approx(0.5 * (math.exp(0.2) - 1), rel=1e-14)
    assert meter >= tv


def test_uniform_c_closed_form():
    for c in (1e-6, 1e-3, 0.3, 2.0):
        lam1 = A.log_a_minus_1(np.log(np.full(7, 1 / 7)), np.full(7, c))
        assert float(A.meter_from_log_am1(lam1)) == pytest.approx(min(1.0, 0.5 * math.expm1(2 * c)), rel=1e-12)
        assert float(A.raw_log_score(lam1)) == pytest.approx(math.log(0.5 * math.expm1(2 * c)), rel=1e-12, abs=1e-12)


def test_theorem1_adversarial_trials_per_query():
    rng = np.random.default_rng(21)
    n_trials = 20_000
    worst = 0.0
    for trial in range(n_trials):
        S = int(rng.integers(2, 40))
        kind = trial % 4
        if kind == 0:      # flat
            logits = np.zeros(S)
        elif kind == 1:    # peaked
            logits = rng.standard_normal(S) * 8
        else:
            logits = rng.standard_normal(S) * rng.uniform(0, 4)
        pt = np.exp(logits - logits.max())
        pt /= pt.sum()
        c = rng.exponential(rng.choice([1e-3, 0.05, 0.5, 3.0]), S)
        if kind == 3:
            c[:] = c[0]  # equal c: the case that breaks the flawed certificate
        sign = rng.choice([-1.0, 1.0], S)
        eps = sign * c * rng.choice([1.0, rng.uniform(0, 1)])
        p = pt * np.exp(-(eps - eps.max()))
        p /= p.sum()
        tv = float(A.total_variation(p, pt))
        meter = float(A.meter_from_log_am1(A.log_a_minus_1(np.log(pt), c)))
        assert meter >= tv * (1 - 1e-12), (trial, meter, tv)
        worst = max(worst, tv / meter if meter > 0 else 0)
    assert worst <= 1.0


def _mp_decode(q, k, kh, vh, w16, sm, s_k=None, tb=None):
    mp.mp.dps = 50
    H, S = q.shape[0], kh.shape[0]
    res = []
    for h in range(H):
        qq = [mp.mpf(float(v)) for v in q[h]]
        xe = [mp.mpf(sm) * mp.fsum(qq[i] * mp.mpf(float(k[t, i])) for i in range(128)) for t in range(S)]
        xc = [mp.mpf(sm) * mp.fsum(qq[i] * mp.mpf(float(kh[t, i])) for i in range(128)) for t in range(S)]
        me, mc = max(xe), max(xc)
        ze = mp.fsum(mp.exp(x - me) for x in xe)
        zc = mp.fsum(mp.exp(x - mc) for x in xc)
        pe = [mp.exp(x - me) / ze for x in xe]
        pc = [mp.exp(x - mc) / zc for x in xc]
        tv = mp.fsum(abs(a - b) for a, b in zip(pe, pc)) / 2
        out = [mp.fsum(pc[t] * mp.mpf(float(vh[t, i])) for t in range(S)) for i in range(128)]
        qb = []
        for b in range(16):
            idx = [4 * b + i for i in range(4)] + [64 + 4 * b + i for i in range(4)]
            qb.append(mp.sqrt(mp.fsum(qq[i] ** 2 for i in idx)))
        c = [mp.mpf(sm) * mp.fsum(qb[b] * mp.mpf(float(w16[t, b])) for b in range(16)) for t in range(S)]
        am1 = mp.fsum(pc[t] * mp.expm1(c[t]) for t in range(S))
        r = dict(tv=tv, out=out, lam1=mp.log(am1) if am1 > 0 else -mp.inf, lse=mc + mp.log(zc))
        if tb is not None:
            dl = mp.mpf(tb["delta_req"]) / (tb["n_layers"] * tb["n_q_heads"] * tb["n_steps"])
            kappa = mp.sqrt(2 * mp.log(2 * S / dl) / 12)
            qn = mp.sqrt(mp.fsum(v * v for v in qq))
            q1 = mp.fsum(abs(mp.mpf(float(x))) for x in q[h])   # the dither grid's bias term, 2^-9 ||q||_1
            u = [mp.mpf(sm) * (qn * kappa + q1 * mp.mpf(2) ** -9) * mp.mpf(float(s_k[t])) for t in range(S)]
            bm1 = mp.fsum(pc[t] * mp.expm1(u[t]) for t in range(S))
            r["lamb"] = mp.log(bm1)
        res.append(r)
    return res


@pytest.mark.parametrize("fmt,S", [("bf16", 2), ("e4m3", 5), ("int8", 8), ("bf16", 8)])
def test_decode_head_brute_force_mpmath(fmt, S):
    rng = np.random.default_rng(31 + S)
    k = rng.standard_normal((S, 128)).astype(np.float32)
    v = rng.standard_normal((S, 128)).astype(np.float32)
    q = rng.standard_normal((3, 128))
    q[1] *= 6.0                     # a peaked head
    q[2] = np.sign(q[2]) * 2.0      # an extreme sign pattern
    xi = dither(5, 0, 0, np.arange(S)[:, None], np.arange(128)[None, :])
    codes, sb, _ = quantize(k, fmt, xi if fmt == "int8" else None)
    kh = dequantize(codes, sb, fmt, xi if fmt == "int8" else None)
    vc, vsb, _ = quantize(v, "e4m3s")
    vh = dequantize(vc, vsb, "e4m3s")
    w16 = fp16_value(witness_bits(kh, k))
    tb = dict(delta_req=1e-3, n_layers=28, n_q_heads=28, n_steps=256) if fmt == "int8" else None
    s_k = fp16_value(sb) if fmt == "int8" else None
    r = A.decode_head(q, k, kh, vh, w16, SM, s_k=s_k, tier_b=tb)
    ref = _mp_decode(q, k, kh, vh, w16, SM, s_k=s_k, tb=tb)
    for h in range(3):
        assert abs(r.tv[h] - float(ref[h]["tv"])) <= 1e-14 + 1e-12 * float(ref[h]["tv"])
        assert np.allclose(r.out[h], [float(x) for x in ref[h]["out"]], rtol=1e-12, atol=1e-14)
        assert r.lse[h] == pytest.approx(float(ref[h]["lse"]), rel=1e-13, abs=1e-13)
        assert r.log_am1_a[h] == pytest.approx(float(ref[h]["lam1"]), abs=1e-11)
        assert r.meter_a[h] >= float(ref[h]["tv"])
        if tb is not None:
            assert r.log_am1_b[h] == pytest.approx(float(ref[h]["lamb"]), abs=1e-11)


def test_theorem2_per_token_and_equality_case():
    rng = np.random.default_rng(41)
    k = rng.standard_normal((256, 128)).astype(np.float32)
    for fmt in ("bf16", "e4m3"):
        codes, _, _ = quantize(k, fmt)
        kh = dequantize(codes, None, fmt)
        r = kh - k.astype(np.float64)
        w16 = fp16_value(witness_bits(kh, k))
        for trial in range(20):
            q = rng.standard_normal(128) * rng.uniform(0.1, 10)
            eps = SM * (r @ q)
            c = A.tier_a_radius(q, w16, SM)
            assert np.all(np.abs(eps) <= c)
    # equality: q_b = lambda_b r_b (lambda_b > 0) and exact (unrounded) band norms
    from oracle.quant import band_norms
    codes, _, _ = quantize(k[:1], "e4m3")
    r = dequantize(codes, None, "e4m3")[0] - k[0].astype(np.float64)
    lam = np.repeat(rng.uniform(0.5, 3, 16), 4)
    q = np.concatenate([r[:64] * lam, r[64:] * lam])
    eps = SM * float(q @ r)
    c_exact = SM * float(band_norms(r) @ A.band_q_norms(q))
    assert eps == pytest.approx(c_exact, rel=1e-12)


def test_identity_quantizer_gives_zero_bound():
    rng = np.random.default_rng(51)
    k = rng.standard_normal((64, 128)).astype(np.float32)
    codes, _, _ = quantize(k, "bf16")
    kb = dequantize(codes, None, "bf16").astype(np.float32)   # bf16-representable keys
    codes2, _, _ = quantize(kb, "bf16")
    kh = dequantize(codes2, None, "bf16")
    w16 = fp16_value(witness_bits(kh, kb))
    q = rng.standard_normal((4, 128))
    r = A.decode_head(q, kb, kh, kh, w16, SM)
    assert np.all(r.log_am1_a == -np.inf)
    assert np.all(r.meter_a == 0.0)
    assert np.all(r.tv == 0.0)


def _rope64(x, pos):
    cos, sin = rope_tables(np.asarray(pos))
    a, b = x[..., :64], x[..., 64:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def test_joint_rope_shift_invariance():
    rng = np.random.default_rng(61)
    S = 48
    k_pre = rng.standard_normal((S, 128))
    rho = rng.standard_normal((S, 128)) * 0.01       # a fixed pre-RoPE residual (black-box quantizer)
    v = rng.standard_normal((S, 128))
    q_pre = rng.standard_normal((2, 128))
    outs = []
    for shift in (0, 1000, 77777):
        pos = np.arange(S) + shift
        k = _rope64(k_pre, pos)
        kh = _rope64(k_pre + rho, pos)
        q = _rope64(q_pre, np.full(2, S + shift))
        from oracle.quant import band_norms
        w = band_norms(kh - k)
        r = A.decode_head(q, k, kh, v, w, SM)
        c = A.tier_a_radius(q[0], w, SM)
        outs.append((r.tv, r.log_am1_a, c))
    for tv, la, c in outs[1:]:
        assert np.allclose(tv, outs[0][0], rtol=1e-9, atol=1e-15)
        assert np.allclose(la, outs[0][1], rtol=0, atol=1e-9)
        assert np.allclose(c, outs[0][2], rtol=1e-12)


def test_lemma2_uniform_mgf():
    from scipy.integrate import quad
    for a in (0.5, 1.0):
        for lam in (0.1, 1.0, 3.0, 8.0):
            num = quad(lambda x: math.exp(lam * x) / (2 * a), -a, a)[0]
            closed = math.sinh(lam * a) / (lam * a)
            assert num == pytest.approx(closed, rel=1e-10)
            assert closed <= math.exp(lam * lam * a * a / 6) * (1 + 1e-15)
    # the dither residual on step s has variance s^2 / 12: the proxy of Lemma 2
    x = np.linspace(-0.5, 0.5, 2_000_001)
    assert np.mean(x * x) == pytest.approx(1 / 12, rel=1e-5)


def test_delta_budget_and_tier_b_constant():
    g = _golden("delta_budget.json")
    den = g["n_layers"] * g["n_q_heads"] * g["n_steps"]
    assert round(den / 1e5, 1) == g["denominator_printed_approx"] / 1e5
    # radius factor: u_t / (sm_scale s_t) = ||q|| sqrt(2 ln(2S/delta_loc)/12) + ||q||_1 2^-9
    kappa = math.sqrt(2 * math.log(2 * 32768 * den / 1e-3) / 12)
    u = A.tier_b_radius(np.ones(128) / math.sqrt(128), np.array([1.0]), 1.0, 32768, 1e-3, 28, 28, 256)
    assert u[0] == pytest.approx(kappa + math.sqrt(128) * 2.0**-9, rel=1e-14)
    # a one-hot query has ||q||_1 = ||q||; the grid term scales with s_t and sm_scale like the rest
    e = np.zeros(128)
    e[37] = -2.0
    u = A.tier_b_radius(e, np.array([0.5, 3.0]), 0.25, 32768, 1e-3, 28, 28, 256)
    assert np.allclose(u, 0.25 * 2.0 * (kappa + 2.0**-9) * np.array([0.5, 3.0]), rtol=1e-14)


def test_tier_b_grid_term_covers_the_dither_bias():
    # the worst case of the grid's bias, built by hand: every channel's input sits where the error mean
    # is largest, and the query's signs follow the bias, so the mean of eps_t is s ||q||_1 2^-9 exactly
    from oracle.philox import subtractive_error_bias_bound
    xi = np.arange(256) * 2.0**-8 - 0.5
    y = np.float32(0.25)                               # on the grid: y + xi hits 1/2 once, rint takes it to 0
    err = np.rint(np.float64(y) + xi) - (np.float64(y) + xi)
    assert err.min() == -0.5 and err.max() == 0.5 - 2.0**-8
    # off the grid by half a step the errors form the symmetric mid-point grid: no bias
    y_mid = np.float64(0.25 + 2.0**-9)
    assert (np.rint(y_mid + xi) - (y_mid + xi)).mean() == 0.0
    mu = err.mean()
    assert abs(mu) == pytest.approx(subtractive_error_bias_bound(), rel=1e-12)
    rng = np.random.default_rng(3)
    q = np.abs(rng.standard_normal(128)) * np.sign(mu)
    s = 0.75
    mean_eps = s * mu * np.sum(q)
    assert abs(mean_eps) == pytest.approx(s * np.sum(np.abs(q)) * 2.0**-9, rel=1e-12)
    u = A.tier_b_radius(q, np.array([s]), 1.0, 1000, 1e-3, 1, 1, 1)
    noise_only = s * np.linalg.norm(q) * math.sqrt(2 * math.log(2 * 1000 / 1e-3) / 12)
    assert u[0] - noise_only == pytest.approx(abs(mean_eps), rel=1e-12)


def test_tier_b_zero_violations_over_dither_seeds():
    rng = np.random.default_rng(71)
    S = 512
    k = rng.standard_normal((S, 128)).astype(np.float32)
    q = rng.standard_normal((4, 128))
    tb = dict(delta_req=1e-2, n_layers=1, n_q_heads=4, n_steps=1)
    viol = 0
    z = []
    for seed in range(200):
        xi = dither(seed, 0, 0, np.arange(S)[:, None], np.arange(128)[None, :])
        codes, sb, _ = quantize(k, "int8", xi)
        kh = dequantize(codes, sb, "int8", xi)
        s = fp16_value(sb)
        eps = SM * ((kh - k.astype(np.float64)) @ q.T)      # [S, 4]
        for h in range(4):
            u = A.tier_b_radius(q[h], s, SM, S, **tb)
            viol += int(np.sum(np.abs(eps[:, h]) > u))
            sig = SM * np.linalg.norm(q[h]) * s / math.sqrt(12)
            z.append(eps[:, h] / sig)
    assert viol == 0
    z = np.concatenate(z)
    assert np.std(z) == pytest.approx(1.0, rel=0.02)   # the proxy equals the variance


def test_proposition1_example():
    g = _golden("proposition1_example.json")
    two = A.two_sided_bound(g["A"], g["A_minus"])
    one = 0.5 * (g["A"] ** 2 - 1)
    assert two > one
    assert two == pytest.approx(0.5 * (2 / 0.6 - 0.6 / 2), rel=1e-15)


def test_split_merge_is_exact():
    rng = np.random.default_rng(81)
    S = 1000
    x = rng.standard_normal(S) * 3
    c = rng.exponential(0.01, S)
    whole = A.log_a_minus_1(x - A.logsumexp(x), c)
    # per-split (lse_s, ln(A_s - 1)) merged with LSE weights
    cuts = [0, 17, 400, 401, 999, 1000]
    lses, lams = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        xs = x[a:b]
        lse = A.logsumexp(xs)
        lses.append(lse)
        lams.append(A.log_a_minus_1(xs - lse, c[a:b]))
    tot = A.logsumexp(np.array(lses))
    merged = A.logsumexp(np.array(lams) + np.array(lses) - tot)
    assert merged == pytest.approx(whole, abs=1e-12)


def test_log_domain_never_overflows():
    lam1 = A.log_a_minus_1(np.log(np.array([0.5, 0.5])), np.array([800.0, 1.0]))
    assert np.isfinite(lam1) and lam1 == pytest.approx(800 + math.log(0.5), rel=1e-12)
    assert float(A.meter_from_log_am1(lam1)) == 1.0
    assert float(A.raw_log_score(lam1)) == pytest.approx(2 * lam1 - math.log(2), rel=1e-12)
