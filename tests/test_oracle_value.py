"""CPU pins of the oracle's value side: the output-error bound and the value witness.

WitCert §3: TV propagates linearly to the attention output,
||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t with rho^v_t = ||v_hat_t - v_t||.
The pins check the oracle's functions against that inequality on random and adversarial cases
(brute force in float64 and in 50-digit arithmetic), against the two cases where each half of the
bound is attained with equality, against the identity quantizer, and the stored fp16 value witness
against its definition (round-up, so never below the exact norms) and against the closed-form
element bound of subtractive dither (|v_hat - v| <= s/2 per element, WitCert §4.2).
"""
import math

import mpmath as mp
import numpy as np
import pytest

from oracle import attention as A
from oracle.encoders import fp16_value
from oracle.philox import dither
from oracle.quant import dequantize, quantize, value_witness_bits, witness_bits

SM = 1.0 / math.sqrt(128)


def _case(rng, S, H=4, key_noise=0.05, val_noise=0.05):
    q = rng.standard_normal((H, 128))
    k = rng.standard_normal((S, 128)).astype(np.float32)
    v = rng.standard_normal((S, 128)).astype(np.float32)
    k_hat = k.astype(np.float64) + key_noise * rng.standard_normal((S, 128))
    v_hat = v.astype(np.float64) + val_noise * rng.standard_normal((S, 128))
    return q, k, v, k_hat, v_hat


def _exact_vw(v_hat, v):
    r = v_hat - v.astype(np.float64)
    return np.stack([np.sqrt((r * r).sum(-1)), np.sqrt((v.astype(np.float64) ** 2).sum(-1))], axis=-1)


@pytest.mark.parametrize("S", [1, 2, 3, 5, 8, 40])
def test_output_bound_holds_random_and_adversarial(S):
    rng = np.random.default_rng(100 + S)
    for trial in range(40):
        q, k, v, k_hat, v_hat = _case(rng, S, key_noise=0.2 * rng.random(), val_noise=0.3 * rng.random())
        if trial % 4 == 1:  # peaked attention on one token
            q[:, :] = 6.0 * k_hat[0] / np.linalg.norm(k_hat[0])
        if trial % 4 == 2:  # values aligned with the sign of p - p~ (first term as large as it gets)
            v = np.ones((S, 128), dtype=np.float32)
            v_hat = v.astype(np.float64).copy()
        w = fp16_value(witness_bits(k_hat, k))
        vw16 = fp16_value(value_witness_bits(v_hat, v))
        res = A.decode_head(q, k, k_hat, v_hat, w, SM, vw=vw16, v_exact=v)
        p_t = np.exp(_log_pt(q, k_hat))
        # decode_head weights the value residuals by the compressed distribution p~ (not p)
        assert np.allclose(res.value_r, p_t @ vw16[:, 0], rtol=1e-12, atol=0)
        assert res.value_vmax == vw16[:, 1].max()
        r_exact, vmax_exact = A.value_side(p_t, _exact_vw(v_hat, v))
        with_tv = A.output_error_bound(res.tv, r_exact, vmax_exact)
        assert np.all(res.out_err <= with_tv * (1 + 1e-12) + 1e-12)
        assert np.all(res.out_err <= res.out_bound_a * (1 + 1e-12) + 1e-12)
        assert np.all(res.meter_a >= res.tv - 1e-15)


def _log_pt(q, k_hat):
    x = SM * (np.asarray(q, np.float64) @ np.asarray(k_hat, np.float64).T)
    return x - A.logsumexp(x)[:, None]


def test_output_bound_mpmath_brute_force():
    """Tiny cases in 50-digit arithmetic: the inequality with the exact TV."""
    mp.mp.dps = 50
    rng = np.random.default_rng(7)
    for _ in range(30):
        S, d = int(rng.integers(1, 5)), 4
        xs = rng.standard_normal(S) * 2
        xh = xs + 0.3 * rng.standard_normal(S)
        v = rng.standard_normal((S, d))
        vh = v + 0.2 * rng.standard_normal((S, d))
        p = [mp.e ** mp.mpf(x) for x in xs]
        zp = mp.fsum(p)
        p = [a / zp for a in p]
        pt = [mp.e ** mp.mpf(x) for x in xh]
        zt = mp.fsum(pt)
        pt = [a / zt for a in pt]
        y = [mp.fsum(p[t] * mp.mpf(v[t, j]) for t in range(S)) for j in range(d)]
        yh = [mp.fsum(pt[t] * mp.mpf(vh[t, j]) for t in range(S)) for j in range(d)]
        err = mp.sqrt(mp.fsum((y[j] - yh[j]) ** 2 for j in range(d)))
        tv = mp.fsum(abs(p[t] - pt[t]) for t in range(S)) / 2
        vmax = max(mp.sqrt(mp.fsum(mp.mpf(v[t, j]) ** 2 for j in range(d))) for t in range(S))
        rho = [mp.sqrt(mp.fsum((mp.mpf(vh[t, j]) - mp.mpf(v[t, j])) ** 2 for j in range(d))) for t in range(S)]
        bound = 2 * tv * vmax + mp.fsum(pt[t] * rho[t] for t in range(S))
        assert err <= bound
        # the oracle's functions give the same bound (in float64)
        r, vm = A.value_side(np.array([[float(a) for a in pt]]),
                             np.stack([[float(a) for a in rho], np.linalg.norm(v, axis=1)], axis=-1))
        got = float(A.output_error_bound(float(tv), r, vm)[0])
        assert abs(got - float(bound)) <= 1e-12 * max(1.0, float(bound))


def test_value_term_equality_when_residuals_align():
    """Exact keys (p = p~, TV = 0) and one common residual vector: ||y - y_hat|| = sum_t p~_t rho^v_t."""
    rng = np.random.default_rng(3)
    q, k, v, _, _ = _case(rng, 12)
    r = 0.1 * rng.standard_normal(128)
    v_hat = v.astype(np.float64) + r[None, :]
    k_hat = k.astype(np.float64)
    w = np.zeros((12, 16))
    res = A.decode_head(q, k, k_hat, v_hat, w, SM, vw=_exact_vw(v_hat, v), v_exact=v)
    assert np.all(res.tv == 0.0) and np.all(res.meter_a == 0.0)
    assert np.allclose(res.out_err, np.linalg.norm(r), rtol=1e-12)
    assert np.allclose(res.out_bound_a, res.out_err, rtol=1e-12)


def test_tv_term_equality_with_sign_aligned_values():
    """Exact values (rho = 0) and v_t = sign(p_t - p~_t) u: ||y - y_hat|| = 2 TV ||u|| exactly."""
    rng = np.random.default_rng(4)
    q, k, _, k_hat, _ = _case(rng, 10, H=1, key_noise=0.3)
    xs = SM * (q @ k.astype(np.float64).T)[0]
    xh = SM * (q @ k_hat.T)[0]
    p, pt = A.softmax(xs), A.softmax(xh)
    u = rng.standard_normal(128)
    v = (np.sign(p - pt)[:, None] * u[None, :]).astype(np.float32)
    u32 = np.abs(v[0]).astype(np.float64)  # |u| after the fp32 rounding, identical for every token
    res = A.decode_head(q, k, k_hat, v.astype(np.float64), np.zeros((10, 16)), SM,
                        vw=_exact_vw(v.astype(np.float64), v), v_exact=v)
    assert np.allclose(res.out_err, 2 * res.tv * np.linalg.norm(u32), rtol=1e-10)
    assert np.allclose(A.output_error_bound(res.tv, res.value_r, res.value_vmax), res.out_err, rtol=1e-10)


def test_identity_quantizers_give_zero_output_bound():
    rng = np.random.default_rng(5)
    q, k, v, _, _ = _case(rng, 9)
    k_hat, v_hat = k.astype(np.float64), v.astype(np.float64)
    w = fp16_value(witness_bits(k_hat, k))
    vw = fp16_value(value_witness_bits(v_hat, v))
    assert np.all(vw[:, 0] == 0.0)
    res = A.decode_head(q, k, k_hat, v_hat, w, SM, vw=vw, v_exact=v)
    assert np.all(res.out_bound_a == 0.0) and np.all(res.out_err == 0.0)


@pytest.mark.parametrize("fmt", ["bf16", "e4m3", "e4m3s", "int8"])
def test_value_witness_rounds_up_within_one_step(fmt):
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 30.0, (64, 1))).astype(np.float32)
    xi = dither(123, 0, 0, np.arange(64)[:, None], np.arange(128)[None, :]) if fmt == "int8" else None
    codes, sb, _ = quantize(v, fmt, xi)
    v_hat = dequantize(codes, sb, fmt, xi)
    vw = fp16_value(value_witness_bits(v_hat, v))
    exact = _exact_vw(v_hat, v)
    assert np.all(vw >= exact)
    # at most one fp16 step above (fp16 keeps 11 significant bits)
    nz = exact > 0
    assert np.all(vw[nz] <= exact[nz] * (1 + 2.0 ** -10) + 2.0 ** -24)
    if fmt == "int8":
        # subtractive dither: every element's reconstruction error is at most s / 2
        s = fp16_value(sb).astype(np.float64)
        assert np.all(exact[:, 0] <= np.sqrt(128) * s / 2 * (1 + 1e-12))


def test_empty_sequence_value_side():
    r, vmax = A.value_side(np.zeros((3, 0)), np.zeros((0, 2)))
    assert r.shape == (3,) and np.all(r == 0.0) and vmax == 0.0
