"""CPU pins of the oracle's fixed-channel outlier bypass (WitCert §6.2.5).

* Table 5 of the page, reproduced qualitatively: with four injected massive RoPE pairs, INT8 dither
  without bypass saturates the meter; bypassing the pairs but leaving them in the amax barely helps;
  bypass plus amax exclusion brings the meter far below the gate threshold (coverage 1 at tau = 0.2).
* Closed forms: the bypassed channels hold fp16_rn(k) and the scale is fp16(fp32(amax_other / 126.5)).
* Element bounds: |k_hat - k| <= s/2 on the INT8 channels (subtractive dither) and
  |k_hat - k| <= 2^-11 |k_hat| + 2^-25 on the bypassed ones (fp16 round to nearest).
* Tier B with the bypass: zero violations of |eps_t| <= u_t over dither seeds; with no bypassed pair
  everything reduces to plain INT8 and plain Tier B.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle.encoders import f32, fp16_bits, fp16_value
from oracle.philox import dither
from oracle.quant import (bypass_channels, dequantize, dequantize_int8_bypass, quantize, quantize_int8_bypass,
                          witness_bits)
from workloads import apply_rope

SM = 1.0 / math.sqrt(128)
PAIRS = [5, 17, 33, 48]


def _keys(S, seed, massive=30.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, 128))
    for j in PAIRS:
        k[:, [j, j + 64]] *= massive
    return apply_rope(k, np.arange(S))


def _raw_meter(q, k32, k_hat):
    w = fp16_value(witness_bits(k_hat, k32))
    res = A.decode_head(q, k32, k_hat, np.zeros_like(k_hat), w, SM)
    return np.exp(res.raw_a)  # 1/2 (A^2 - 1), unclamped


def test_table5_bypass_needs_amax_exclusion():
    S, H = 256, 8
    meters = {"none": [], "bypass_only": [], "bypass_excl": []}
    for seed in range(3):
        k32 = _keys(S, 100 + seed)
        q = np.random.default_rng(200 + seed).standard_normal((H, 128))
        xi = dither(seed, 0, 0, np.arange(S)[:, None], np.arange(128)[None, :])
        codes, sb, _ = quantize(k32, "int8", xi)
        meters["none"].append(_raw_meter(q, k32, dequantize(codes, sb, "int8", xi)))
        for name, excl in (("bypass_only", False), ("bypass_excl", True)):
            c, s_, ob, valid = quantize_int8_bypass(k32, xi, PAIRS, exclude_from_amax=excl)
            assert np.all(valid)
            meters[name].append(_raw_meter(q, k32, dequantize_int8_bypass(c, s_, ob, xi, PAIRS)))
    med = {k: float(np.median(np.concatenate(v))) for k, v in meters.items()}
    assert med["none"] >= 1.0                                   # saturated: coverage 0 at tau = 0.2
    assert abs(med["bypass_only"] - med["none"]) <= 0.3 * med["none"]   # bypass alone barely helps
    assert med["bypass_excl"] <= med["none"] / 10                # an order of magnitude and more lower
    assert np.max(np.concatenate(meters["bypass_excl"])) < 0.2   # coverage 1 at tau = 0.2


def test_bypass_closed_forms():
    k32 = _keys(64, 7)
    xi = dither(9, 2, 1, np.arange(64)[:, None], np.arange(128)[None, :])
    codes, sb, ob, valid = quantize_int8_bypass(k32, xi, PAIRS)
    ch = bypass_channels(PAIRS)
    assert list(ch) == [5, 69, 17, 81, 33, 97, 48, 112]
    assert np.array_equal(ob, fp16_bits(k32[:, ch].astype(np.float64), "rne"))
    assert np.all(codes[:, ch] == 0)
    other = np.delete(np.abs(k32), ch, axis=1).max(axis=1)
    expect = fp16_bits(f32(other.astype(np.float64) / 126.5), "rne")
    assert np.array_equal(sb, expect)
    # the INT8 channels are exactly plain dithered INT8 with that scale
    plain_codes, _, _ = quantize(np.where(np.isin(np.arange(128), ch), 0, k32).astype(np.float32), "int8", xi)
    keep = ~np.isin(np.arange(128), ch)
    # the plain quantizer's amax over the zeroed-out row equals the bypass amax, so the codes agree
    assert np.array_equal(codes[:, keep], plain_codes[:, keep])


def test_bypass_element_bounds():
    k32 = _keys(128, 8, massive=300.0)
    xi = dither(3, 0, 0, np.arange(128)[:, None], np.arange(128)[None, :])
    codes, sb, ob, _ = quantize_int8_bypass(k32, xi, PAIRS)
    kh = dequantize_int8_bypass(codes, sb, ob, xi, PAIRS)
    r = np.abs(kh - k32.astype(np.float64))
    ch = bypass_channels(PAIRS)
    keep = ~np.isin(np.arange(128), ch)
    s = fp16_value(sb)[:, None]
    assert np.all(r[:, keep] <= s / 2 * (1 + 1e-12))
    assert np.all(r[:, ch] <= A.FP16_REL * np.abs(kh[:, ch]) + A.FP16_ABS)


def test_fp16_rounding_bound_over_ranges():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-1, 1, 200000) * 10.0 ** rng.uniform(-9, 4.8, 200000),
                        np.arange(-2048, 2048) * 2.0 ** -24 * 0.73])
    x = x.astype(np.float32).astype(np.float64)
    rn = fp16_value(fp16_bits(x, "rne"))
    ok = np.isfinite(rn)
    assert np.all(np.abs(rn[ok] - x[ok]) <= A.FP16_REL * np.abs(rn[ok]) + A.FP16_ABS)


def test_tier_b_with_bypass_zero_violations():
    S, H, L, T, dreq = 300, 4, 28, 256, 1e-2
    k32 = _keys(S, 11, massive=25.0)
    q = np.random.default_rng(12).standard_normal((H, 128))
    ch = bypass_channels(PAIRS)
    viol = 0
    for seed in range(40):
        xi = dither(1000 + seed, 0, 0, np.arange(S)[:, None], np.arange(128)[None, :])
        codes, sb, ob, _ = quantize_int8_bypass(k32, xi, PAIRS)
        kh = dequantize_int8_bypass(codes, sb, ob, xi, PAIRS)
        s_k = fp16_value(sb)
        for h in range(H):
            eps = SM * (q[h] @ (kh - k32.astype(np.float64)).T)
            u = A.tier_b_radius_bypass(q[h], s_k, fp16_value(ob), ch, SM, S, dreq, L, H, T)
            viol += int(np.sum(np.abs(eps) > u))
    assert viol == 0


def test_no_pairs_reduces_to_plain_int8():
    k32 = _keys(40, 13, massive=1.0)
    xi = dither(5, 1, 2, np.arange(40)[:, None], np.arange(128)[None, :])
    c0, s0, _ = quantize(k32, "int8", xi)
    c1, s1, ob, _ = quantize_int8_bypass(k32, xi, [])
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1) and ob.shape == (40, 0)
    q = np.random.default_rng(3).standard_normal(128)
    u0 = A.tier_b_radius(q, fp16_value(s0), SM, 40, 1e-2, 1, 1, 256)
    u1 = A.tier_b_radius_bypass(q, fp16_value(s1), fp16_value(ob), bypass_channels([]), SM, 40, 1e-2, 1, 1, 256)
    assert np.array_equal(u0, u1)
