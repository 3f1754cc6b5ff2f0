"""Pins of the oracle's quantizers and witness (CPU).

What pins what:
* INT8 dither: |x_hat - x| <= s/2 (up to the binary32 rounding of x/s + xi)
  and no code clips (WitCert §4.2 and the §6.2.1 acceptance items);
  the scale is the fp16 rounding of amax/126.5 (closed form); the stored scale
  is the one quantized with (a row whose amax makes fp32 and fp16 scales differ).
* E4M3 scaled: reconstruction error <= half an E4M3 step at each value.
* BF16 keys: residual <= 2^-9 relative; bf16-representable keys give witness 0.
* Witness and value witness: the smallest fp16 at or above the exact norm, equal
  to a binary search in exact rationals on random rows (binary32 subnormals to
  1e35), on near-ties built to defeat the float64 bracket (h^2 + tiny, exact
  squares, a 3-4-5 triple), at the overflow edge and for non-finite rows; band
  membership by RoPE pairs.
* Lemma 1 (RoPE band unitarity): the band norms of a rotated residual equal
  those of the unrotated one.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle.encoders import e4m3_value, fp16_value
from oracle.philox import dither
from oracle.quant import band_norms, band_of_channel, dequantize, quantize, witness_bits
from workloads import apply_rope


def _rows(n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, 128)) * scale).astype(np.float32)


def test_band_membership_half_split():
    b = band_of_channel(np.arange(128))
    for band in range(16):
        idx = np.where(b == band)[0]
        assert list(idx) == [4 * band + i for i in range(4)] + [64 + 4 * band + i for i in range(4)]


@pytest.mark.parametrize("scale", [1.0, 0.01, 37.0])
def test_int8_dither_error_bound_and_no_clipping(scale):
    x = _rows(4096, 1, scale)
    xi = dither(7, 0, 0, np.arange(4096)[:, None], np.arange(128)[None, :])
    codes, sb, valid = quantize(x, "int8", xi)
    assert valid.all()
    s = fp16_value(sb)
    # scale closed form: fp16(fp32(amax / 126.5))
    amax = np.abs(x).max(axis=1).astype(np.float64)
    t = (amax / 126.5).astype(np.float32).astype(np.float64)
    assert np.array_equal(s, t.astype(np.float16).astype(np.float64))
    xh = dequantize(codes, sb, "int8", xi)
    err = np.abs(xh - x.astype(np.float64)) / s[:, None]
    # fp32 rounding of x/s and of + xi can move the rounding point by ~2^-17 code units
    assert err.max() <= 0.5 + 2**-16
    # no clipping: the unclamped nearest integer of x/s + xi is inside [-127, 127]
    y2 = (x.astype(np.float64) / s[:, None]).astype(np.float32).astype(np.float64) + xi
    assert np.abs(np.rint(y2)).max() <= 127


def test_int8_zero_row_and_stored_scale_rule():
    x = np.zeros((2, 128), dtype=np.float32)
    x[1, 5] = 1.0
    xi = dither(1, 0, 0, np.arange(2)[:, None], np.arange(128)[None, :])
    codes, sb, _ = quantize(x, "int8", xi)
    assert sb[0] == 0 and np.all(codes[0] == 0)
    # amax = 1: fp32(1/126.5) differs from its fp16 rounding; codes use the fp16 value
    s16 = fp16_value(sb[1])
    assert s16 != np.float32(1 / 126.5)
    y = np.float32(np.float64(np.float32(1.0)) / s16)
    assert codes[1, 5] == int(np.clip(np.rint(np.float64(np.float32(np.float64(y) + xi[1, 5]))), -127, 127))


def test_e4m3_scaled_error_and_scale():
    v = _rows(2048, 2, 3.0)
    codes, sb, valid = quantize(v, "e4m3s")
    assert valid.all()
    s = fp16_value(sb)
    amax = np.abs(v).max(axis=1).astype(np.float64)
    assert np.array_equal(s, (amax / 448).astype(np.float32).astype(np.float64).astype(np.float16).astype(np.float64))
    vh = dequantize(codes, sb, "e4m3s")
    y = v.astype(np.float64) / s[:, None]
    # half an E4M3 step at |y| (step 2^(e-3), e = exponent of |y|, at least 2^-9)
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0**-6)))
    step = 2.0 ** (e - 3)
    assert np.all(np.abs(vh / s[:, None] - y) <= step / 2 * (1 + 1e-6) + np.maximum(np.abs(y) - 448, 0))


def test_bf16_residual_and_identity_quantizer():
    k = _rows(1024, 3)
    codes, _, _ = quantize(k, "bf16")
    kh = dequantize(codes, None, "bf16")
    assert np.all(np.abs(kh - k) <= np.abs(k) * 2.0**-8 + 1e-45)
    # keys that are already bfloat16 values have zero residual and zero witness
    w = witness_bits(kh, kh.astype(np.float32))
    assert np.all(fp16_value(w) == 0.0)


def test_witness_is_round_up_of_exact_band_norm():
    k = _rows(64, 4)
    xi = dither(3, 1, 0, np.arange(64)[:, None], np.arange(128)[None, :])
    for fmt in ("bf16", "e4m3", "int8"):
        codes, sb, _ = quantize(k, fmt, xi if fmt == "int8" else None)
        kh = dequantize(codes, sb, fmt, xi if fmt == "int8" else None)
        w = witness_bits(kh, k)
        wv = fp16_value(w)
        for t in range(0, 64, 7):
            r = [Fraction(float(a)) - Fraction(float(b)) for a, b in zip(kh[t], k[t].astype(np.float64))]
            for b in range(16):
                idx = [4 * b + i for i in range(4)] + [64 + 4 * b + i for i in range(4)]
                n2 = sum(r[i] * r[i] for i in idx)
                up = Fraction(float(wv[t, b]))
                assert up * up >= n2, (fmt, t, b)
                below = np.nextafter(np.float16(wv[t, b]), np.float16(0)).astype(np.float64)
                if wv[t, b] > 0:
                    assert Fraction(float(below)) ** 2 < n2, (fmt, t, b)


def test_lemma1_band_norms_invariant_under_rope():
    rng = np.random.default_rng(5)
    r = rng.standard_normal((32, 128))
    base = band_norms(r)
    for pos in (0, 1, 517, 131071):
        # rotate the residual in float64 (apply_rope rounds to binary32, so use its float64 math here)
        from workloads import rope_tables
        cos, sin = rope_tables(np.full(32, pos))
        a, b = r[:, :64], r[:, 64:]
        rr = np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)
        assert np.allclose(band_norms(rr), base, rtol=1e-13, atol=0)
    # and the binary32 rotation used for the inputs changes them only at binary32 precision
    assert np.allclose(band_norms(apply_rope(r, np.full(32, 99))), base, rtol=1e-6)


def test_nonfinite_and_overflow_rows_flagged():
    x = _rows(3, 6)
    x[0, 0] = np.nan
    x[1, 0] = 3.0e7  # amax / 126.5 overflows fp16
    xi = np.zeros((3, 128))
    _, _, valid = quantize(x, "int8", xi)
    assert list(valid) == [False, False, True]
    _, _, valid = quantize(x, "e4m3s")
    # 3e7 / 448 = 66,964 is past the fp16 round-to-nearest overflow threshold 65,520
    assert list(valid) == [False, False, True]


# ------------------------------------------------------------------ exact norms rounded up to fp16
def _fp16_ru_norm_brute(a_hat, a):
    """The definition in exact rationals: the smallest non-negative binary16 value (bit pattern) whose
    square is at least sum (a_hat - a)^2; +inf (0x7C00) when none is."""
    t = sum((Fraction(float(u)) - Fraction(float(v))) ** 2 for u, v in zip(a_hat, a))
    lo, hi = 0, 0x7C00        # binary search over the increasing positive binary16 patterns
    while lo < hi:
        mid = (lo + hi) // 2
        h = Fraction(float(np.uint16(mid).view(np.float16)))
        if h * h >= t:
            hi = mid
        else:
            lo = mid + 1
    return lo


def _brute_rows(xh, x):
    return np.array([_fp16_ru_norm_brute(u, v) for u, v in zip(xh.reshape(-1, xh.shape[-1]),
                                                               x.reshape(-1, x.shape[-1]))]).reshape(xh.shape[:-1])


@pytest.mark.parametrize("n", [1, 8, 128])
def test_exact_norm_matches_rational_brute_force(n):
    from oracle.quant import norm_fp16_ru_bits

    rng = np.random.default_rng(n)
    rows = 300 if n < 128 else 60
    # magnitudes from binary32 subnormals to 1e35, mixed within rows
    mag = 10.0 ** rng.uniform(-44, 35, (rows, n))
    x = (rng.standard_normal((rows, n)) * mag).astype(np.float32).astype(np.float64)
    xh = np.where(rng.random((rows, n)) < 0.5, x, (x * (1 + rng.standard_normal((rows, n)) * 1e-3)).astype(np.float32))
    got = norm_fp16_ru_bits(xh, x)
    assert np.array_equal(got, _brute_rows(xh, x))


def test_exact_norm_decides_near_ties_exactly():
    """Rows whose float64 bracket holds an fp16 square: the answer still follows the exact sum."""
    from oracle.quant import norm_fp16_ru_bits

    cases, want = [], []
    for hb in (0x0001, 0x03FF, 0x1C00, 0x3555, 0x3C00, 0x7BFE):
        h = float(np.uint16(hb).view(np.float16))
        tiny = h * 2.0 ** -70
        cases.append([h, tiny, 0.0]); want.append(hb + 1)     # h^2 + tiny^2 > h^2: the next fp16 value
        cases.append([h, 0.0, 0.0]); want.append(hb)          # exactly h
        cases.append([0.0, h, 0.0]); want.append(hb)
    # 3-4-5: (3u)^2 + (4u)^2 = (5u)^2 exactly
    u = 2.0 ** -12
    cases.append([3 * u, 4 * u, 0.0]); want.append(int(np.float16(5 * u).view(np.uint16)))
    cases.append([3 * u, 4 * u, u * 2.0 ** -40]); want.append(int(np.float16(5 * u).view(np.uint16)) + 1)
    cases.append([0.0, 0.0, 0.0]); want.append(0)
    cases.append([65504.0, 0.0, 0.0]); want.append(0x7BFF)
    cases.append([65504.0, 1e-3, 0.0]); want.append(0x7C00)   # above the largest finite: +inf
    cases.append([2.0 ** -149, 0.0, 0.0]); want.append(1)     # any positive norm below 2^-24 rounds up to it
    xh = np.array(cases)
    got = norm_fp16_ru_bits(xh, np.zeros_like(xh))
    assert list(got) == want
    assert np.array_equal(got, _brute_rows(xh, np.zeros_like(xh)))
    # the same as residuals of nearby binary32 pairs (the difference itself carries the small term)
    a = np.float64(np.float32(1.0 + 2.0 ** -20))
    r = a - 1.0                       # 2^-20, an fp16 value
    xh2 = np.array([[a, 1.0 + 2.0 ** -23, 2.0 ** -60]])
    x2 = np.array([[1.0, 1.0, 0.0]])
    assert np.array_equal(norm_fp16_ru_bits(xh2, x2), _brute_rows(xh2, x2))
    assert norm_fp16_ru_bits(np.array([[a]]), np.array([[1.0]]))[0] == np.float16(r).view(np.uint16)


def test_witness_and_value_witness_are_exact_norms():
    from oracle.quant import value_witness_bits

    k = _rows(40, 8)
    xi = dither(5, 2, 1, np.arange(40)[:, None], np.arange(128)[None, :])
    codes, sb, _ = quantize(k, "int8", xi)
    kh = dequantize(codes, sb, "int8", xi)
    w = witness_bits(kh, k)
    bands = [[4 * b + i for i in range(4)] + [64 + 4 * b + i for i in range(4)] for b in range(16)]
    for t in range(0, 40, 9):
        assert [int(v) for v in w[t]] == [_fp16_ru_norm_brute(kh[t, idx], k[t, idx].astype(np.float64))
                                          for idx in bands]
    vw = value_witness_bits(kh, k)
    for t in range(0, 40, 13):
        assert int(vw[t, 0]) == _fp16_ru_norm_brute(kh[t], k[t].astype(np.float64))
        assert int(vw[t, 1]) == _fp16_ru_norm_brute(k[t].astype(np.float64), np.zeros(128))
    # a non-finite row gives the NaN pattern (the library flags such rows)
    bad = k.copy()
    bad[0, 5] = np.inf                     # channel 5 lies in band 1
    wb = witness_bits(kh, bad)
    assert wb[0, 1] == 0x7E00 and np.array_equal(np.delete(wb[0], 1), np.delete(w[0], 1))
