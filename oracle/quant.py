"""Quantize-on-append, dequantization and the band-norm witness (oracle; test infrastructure).

Layouts ("Compress the shared cartridge", table "Keys carry the cartridge
quantization loss"; WitCert §4.2 and §6.2.3):

  'bf16'   BF16 code, round-to-nearest-even (the K16 half of K16/V8 and K16/V16)
  'e4m3'   raw FP8 E4M3 cast, no scale (the K8/V8 raw-cast layout)
  'e4m3s'  FP8 E4M3 with one fp16 scale per (token, kv head): s = fp16(amax/448)
  'int8'   subtractively dithered INT8 with one fp16 scale per (token, kv head):
           s = fp16(amax/126.5), code = rint(x/s + xi), x_hat = s*(code - xi)

Rules taken from the pages
--------------------------
* WitCert §4.2 "Subtractive dither": x_hat = s*(round(x/s + xi) - xi), xi uniform
  on [-1/2, 1/2), s = amax/(Q - 1/2) with Q = 127, i.e. amax/126.5, chosen so that
  no code clips.
* WitCert §6.2.1: quantization must use the *stored* fp16 scale, not the fp32
  one it was rounded from.
* WitCert §6.2.3: with token-granular paging the scale is per token (per
  channel group); the workloads here use one group of 128 channels per
  (token, kv head).  ``quantize_int8_groups`` is the page's default granularity,
  one fp16 scale per token per group of G_c = 32 channels (§6.2.3, Table 4);
  each group follows the INT8 rules above with its own amax.
* WitCert §4.1, eq. (2): the witness w_{t,b} = ||r_{t,b}|| is the Euclidean
  norm of the key residual r = k_hat - k over band b, stored in fp16.  Bands are
  B = 16 contiguous groups of RoPE frequency pairs (4 pairs = 8 coordinates each).
* WitCert §6.2.5 (fixed-channel outlier bypass): a fixed set of m RoPE pairs per
  (layer, kv head) keeps its 2m key channels in fp16, and those channels are
  excluded from the group amax (bypassing without the exclusion leaves the scale,
  and so the error of every other channel, unchanged).  Here the INT8 code of a
  bypassed channel is 0 and its value is the fp16 one (round to nearest even).
* WitCert §3 (the output bound ||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t):
  the value side needs, per token, rho^v_t = ||v_hat_t - v_t|| and ||v_t||; stored
  here as a value witness of two fp16 numbers per (token, kv head).

Readings where the pages are silent
-----------------------------------
* RoPE pairs are half-split: pair j = coordinates (j, j + 64).  Band b therefore
  holds coordinates 4b..4b+3 and 64+4b..64+4b+3.
* Every scalar step is the binary32 operation (evaluated in float64 and rounded
  once): t = fp32(amax / 126.5) (or / 448), s = fp16_rn(t), y = fp32(x / s),
  y2 = fp32(y + xi), code = clamp(round_half_even(y2), -127, 127).
* amax = 0 (or a scale that rounds to fp16 zero) stores scale 0 and all-zero codes.
* The fp16 witness is the exact residual norm rounded up, so it never under-states
  it: the smallest binary16 value whose square is at least the exact sum of squares.
* FP8-scaled values use s = fp16_rn(fp32(amax / 448)) and code = e4m3(fp32(v / s))
  (round-to-nearest-even, saturating at +-448).
* A channel group is G_c contiguous channels in storage order, group g = channels
  [g G_c, (g + 1) G_c); with half-split RoPE a pair's two channels fall in groups
  g and g + 64 / G_c.  The scales of a row are stored group by group.
"""
from __future__ import annotations

import numpy as np

from .encoders import (
    bf16_bits_rne,
    bf16_value,
    e4m3_bits_rne_satfinite,
    e4m3_value,
    f32,
    fp16_bits,
    fp16_value,
)

__all__ = [
    "FORMATS",
    "HEAD_DIM",
    "N_BANDS",
    "band_of_channel",
    "quantize",
    "dequantize",
    "witness_bits",
    "value_witness_bits",
    "bypass_channels",
    "quantize_int8_bypass",
    "dequantize_int8_bypass",
    "quantize_int8_groups",
    "dequantize_int8_groups",
    "band_norms",
    "norm_fp16_ru_bits",
]

HEAD_DIM = 128
N_BANDS = 16
FORMATS = ("bf16", "e4m3", "e4m3s", "int8")
INT8_QMAX = 127
INT8_DIVISOR = 126.5  # Q - 1/2 with Q = 127
E4M3_DIVISOR = 448.0


def band_of_channel(c):
    """Band index of head-dim coordinate ``c`` under half-split RoPE pairing with 16 bands."""
    c = np.asarray(c)
    return (c % (HEAD_DIM // 2)) // ((HEAD_DIM // 2) // N_BANDS)


def _scale_bits(amax32: np.ndarray, divisor: float) -> np.ndarray:
    t = f32(amax32.astype(np.float64) / divisor)
    return fp16_bits(t.astype(np.float64), "rne")


def quantize(x32: np.ndarray, fmt: str, xi: np.ndarray | None = None):
    """Quantize rows of 128 binary32 values.

    ``x32``: [..., 128] float32.  ``xi``: [..., 128] dither (float64, exact) for
    'int8'.  Returns ``(codes, scale_bits, valid)``: codes as uint16 (bf16
    patterns), uint8 (e4m3 patterns) or int8 (INT8 codes); scale_bits [...]
    uint16 fp16 patterns or None; ``valid`` [...] False where the row holds a
    non-finite value or its scale overflows fp16 (the library flags those rows).
    """
    x = np.asarray(x32, dtype=np.float32)
    assert x.shape[-1] == HEAD_DIM
    finite = np.all(np.isfinite(x), axis=-1)
    if fmt == "bf16":
        return bf16_bits_rne(x), None, finite
    if fmt == "e4m3":
        return e4m3_bits_rne_satfinite(x), None, finite
    amax = np.max(np.abs(x), axis=-1)
    if fmt == "e4m3s":
        s_bits = _scale_bits(amax, E4M3_DIVISOR)
        s = fp16_value(s_bits)
        valid = finite & np.isfinite(s)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = f32(x.astype(np.float64) / s[..., None])
        codes = e4m3_bits_rne_satfinite(y)
        codes = np.where((s == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
        return codes, s_bits, valid
    if fmt == "int8":
        assert xi is not None and xi.shape == x.shape
        s_bits = _scale_bits(amax, INT8_DIVISOR)
        s = fp16_value(s_bits)
        valid = finite & np.isfinite(s)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = f32(x.astype(np.float64) / s[..., None])
            y2 = f32(y.astype(np.float64) + xi)
            code = np.clip(np.rint(y2.astype(np.float64)), -INT8_QMAX, INT8_QMAX)
        code = np.where((s == 0)[..., None] | ~np.isfinite(code), 0, code)
        return code.astype(np.int8), s_bits, valid
    raise ValueError(fmt)


def bypass_channels(pairs) -> np.ndarray:
    """Key channels of outlier RoPE pairs j (half-split pairing: channels j and j + 64), in the stored
    column order: column 2i -> channel pairs[i], column 2i + 1 -> channel pairs[i] + 64."""
    pairs = np.asarray(pairs, dtype=np.int64)
    assert pairs.ndim == 1 and np.all((pairs >= 0) & (pairs < HEAD_DIM // 2)) and len(set(pairs.tolist())) == len(pairs)
    return np.stack([pairs, pairs + HEAD_DIM // 2], axis=-1).reshape(-1)


def quantize_int8_bypass(x32: np.ndarray, xi: np.ndarray, pairs, exclude_from_amax: bool = True):
    """Subtractively dithered INT8 with the fixed-channel outlier bypass (WitCert §6.2.5).

    Returns ``(codes, scale_bits, outlier_bits, valid)``: INT8 codes (0 at bypassed channels), the fp16
    scale of amax over the other channels (over all channels when ``exclude_from_amax`` is False, the
    page's "bypass, amax unchanged" control), the fp16 patterns [..., 2m] of the bypassed channels in
    column order, and ``valid`` (False for non-finite input or an fp16 overflow of scale or outlier).
    """
    x = np.asarray(x32, dtype=np.float32)
    ch = bypass_channels(pairs)
    keep = np.ones(HEAD_DIM, dtype=bool)
    keep[ch] = False
    finite = np.all(np.isfinite(x), axis=-1)
    amax = np.max(np.abs(np.where(keep, x, 0.0) if exclude_from_amax else x), axis=-1).astype(np.float32)
    s_bits = _scale_bits(amax, INT8_DIVISOR)
    s = fp16_value(s_bits)
    out_bits = fp16_bits(x[..., ch].astype(np.float64), "rne")
    valid = finite & np.isfinite(s) & np.all(np.isfinite(fp16_value(out_bits)), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = f32(x.astype(np.float64) / s[..., None])
        y2 = f32(y.astype(np.float64) + xi)
        code = np.clip(np.rint(y2.astype(np.float64)), -INT8_QMAX, INT8_QMAX)
    code = np.where((s == 0)[..., None] | ~np.isfinite(code) | ~keep, 0, code)
    return code.astype(np.int8), s_bits, out_bits, valid


def dequantize_int8_bypass(codes, scale_bits, outlier_bits, xi, pairs) -> np.ndarray:
    """x_hat: s (code - xi) on the INT8 channels, the fp16 value on the bypassed ones."""
    xh = dequantize(codes, scale_bits, "int8", xi)
    xh[..., bypass_channels(pairs)] = fp16_value(outlier_bits)
    return xh


def quantize_int8_groups(x32: np.ndarray, xi: np.ndarray, group: int = 32):
    """Subtractively dithered INT8 with one fp16 scale per token per group of ``group`` contiguous
    channels (WitCert §6.2.3, Table 4: token x G_c-channel groups, G_c = 32 by default).

    Every group is quantized as its own row: s_g = fp16_rn(fp32(amax_g / 126.5)), y = fp32(x / s_g),
    y2 = fp32(y + xi), code = clamp(round_half_even(y2), -127, 127); a group whose scale is 0 stores
    all-zero codes.  Returns ``(codes [..., 128] int8, scale_bits [..., 128 / group] uint16, valid [...])``,
    ``valid`` False for a non-finite input or any group scale that overflows fp16.
    """
    x = np.asarray(x32, dtype=np.float32)
    assert x.shape[-1] == HEAD_DIM and HEAD_DIM % group == 0 and xi.shape == x.shape
    n_groups = HEAD_DIM // group
    xg = x.reshape(x.shape[:-1] + (n_groups, group))
    finite = np.all(np.isfinite(x), axis=-1)
    s_bits = _scale_bits(np.max(np.abs(xg), axis=-1), INT8_DIVISOR)
    s = fp16_value(s_bits)
    valid = finite & np.all(np.isfinite(s), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = f32(xg.astype(np.float64) / s[..., None])
        y2 = f32(y.astype(np.float64) + np.asarray(xi, dtype=np.float64).reshape(xg.shape))
        code = np.clip(np.rint(y2.astype(np.float64)), -INT8_QMAX, INT8_QMAX)
    code = np.where((s == 0)[..., None] | ~np.isfinite(code), 0, code)
    return code.reshape(x.shape).astype(np.int8), s_bits, valid


def dequantize_int8_groups(codes: np.ndarray, scale_bits: np.ndarray, xi: np.ndarray) -> np.ndarray:
    """x_hat_c = s_{g(c)} (code_c - xi_c), g(c) = c // G_c with G_c = 128 / scale_bits.shape[-1] (exact)."""
    group = HEAD_DIM // scale_bits.shape[-1]
    s = np.repeat(fp16_value(scale_bits), group, axis=-1)
    return s * (np.asarray(codes).astype(np.float64) - np.asarray(xi, dtype=np.float64))


def dequantize(codes: np.ndarray, scale_bits: np.ndarray | None, fmt: str, xi: np.ndarray | None = None):
    """Exact float64 reconstruction x_hat of stored codes."""
    if fmt == "bf16":
        return bf16_value(codes)
    if fmt == "e4m3":
        return e4m3_value(codes)
    s = fp16_value(scale_bits)[..., None]
    if fmt == "e4m3s":
        return s * e4m3_value(codes)
    if fmt == "int8":
        # s (11 bits) * (code - xi) (at most 31 bits) is exact in float64
        return s * (codes.astype(np.float64) - xi)
    raise ValueError(fmt)


def band_norms(r: np.ndarray) -> np.ndarray:
    """Per-band Euclidean norms of residual rows r [..., 128] -> [..., 16] float64."""
    r = np.asarray(r, dtype=np.float64)
    half = HEAD_DIM // 2
    per = half // N_BANDS
    lo = r[..., :half].reshape(r.shape[:-1] + (N_BANDS, per))
    hi = r[..., half:].reshape(r.shape[:-1] + (N_BANDS, per))
    return np.sqrt(np.sum(lo * lo, axis=-1) + np.sum(hi * hi, axis=-1))


_SQ16 = None


def _fp16_squares() -> np.ndarray:
    """h * h for every non-negative binary16 value h, in bit-pattern order 0x0000 .. 0x7C00 (+inf last).

    Positive binary16 values increase with their bit pattern, and the square of a value with 11
    significant bits is exact in float64, so the table is an exact, increasing list of squares.
    """
    global _SQ16
    if _SQ16 is None:
        h = fp16_value(np.arange(0x7C01, dtype=np.uint16))
        _SQ16 = h * h
    return _SQ16


def norm_fp16_ru_bits(a_hat: np.ndarray, a: np.ndarray) -> np.ndarray:
    """binary16 pattern of ||a_hat - a|| over the last axis, rounded up, of the EXACT norm.

    The result is the smallest non-negative binary16 value h (+inf above 65504) with
    h^2 >= sum_i (a_hat_i - a_i)^2, the sum taken in exact arithmetic.  a_hat and a hold exact
    values (a binary32 input, a decoded code).  Rows with a non-finite input give the NaN pattern.

    The comparison is made first against a float64 bracket [T_lo, T_hi] of the exact sum of
    squares (TwoSum gives each difference exactly as d + e; the relative error of sum d^2 is below
    (n + 4) 2^-52 for n terms; the bracket is twice that wide).  A row whose bracket holds no
    binary16 square between h's predecessor and h is decided by it; any other row is decided in
    exact rational arithmetic (``fractions.Fraction``).
    """
    x = np.asarray(a_hat, dtype=np.float64)
    y = np.asarray(a, dtype=np.float64)
    x, y = np.broadcast_arrays(x, y)
    n = x.shape[-1]
    finite = np.all(np.isfinite(x) & np.isfinite(y), axis=-1)
    xs = np.where(np.isfinite(x) & np.isfinite(y), x, 0.0)
    ys = np.where(np.isfinite(x) & np.isfinite(y), y, 0.0)
    d = xs - ys
    # TwoSum(xs, -ys): d + e == xs - ys exactly
    bp = d - xs
    e = (xs - (d - bp)) + (-ys - bp)
    exact_zero = np.all((d == 0) & (e == 0), axis=-1)
    T = np.sum(d * d, axis=-1)
    eps = (n + 4) * 2.0 ** -52
    t_lo, t_hi = T * (1.0 - 2 * eps), T * (1.0 + 2 * eps)
    sq = _fp16_squares()
    hi = np.searchsorted(sq, t_hi, side="left")
    lo = np.searchsorted(sq, t_lo, side="left")
    out = hi.astype(np.int64)
    pred = np.maximum(hi - 1, 0)
    decided = (hi == 0) | (sq[pred] < t_lo)
    out = np.where(exact_zero, 0, out)
    todo = np.flatnonzero(~decided & ~exact_zero & finite)
    if todo.size:
        from fractions import Fraction

        shape = out.shape
        out = out.reshape(-1)
        flat_x, flat_y = xs.reshape(-1, n), ys.reshape(-1, n)
        lo_f, hi_f = lo.reshape(-1), hi.reshape(-1)
        for i in todo:
            t_exact = sum((Fraction(float(u)) - Fraction(float(v))) ** 2 for u, v in zip(flat_x[i], flat_y[i]))
            k = int(lo_f[i])   # the answer lies in [lo, hi]: sq[lo - 1] < t_lo <= t_exact <= t_hi <= sq[hi]
            while k < int(hi_f[i]) and Fraction(float(sq[k])) < t_exact:
                k += 1
            out[i] = k
        out = out.reshape(shape)
    out = np.where(finite, out, 0x7E00)
    return out.astype(np.uint16)


def _band_view(x: np.ndarray) -> np.ndarray:
    """[..., 128] -> [..., 16 bands, 8]: band b holds channels 4b..4b+3 and 64+4b..64+4b+3."""
    half = HEAD_DIM // 2
    per = half // N_BANDS
    lo = x[..., :half].reshape(x.shape[:-1] + (N_BANDS, per))
    hi = x[..., half:].reshape(x.shape[:-1] + (N_BANDS, per))
    return np.concatenate([lo, hi], axis=-1)


def value_witness_bits(v_hat: np.ndarray, v32: np.ndarray) -> np.ndarray:
    """Value witness [..., 2] fp16 (round-up) patterns: (||v_hat - v||, ||v||) over the 128 channels, each
    the exact norm rounded up, so that neither the value reconstruction error nor the value norm is
    under-stated."""
    v = np.asarray(v32, dtype=np.float32).astype(np.float64)
    vh = np.asarray(v_hat, dtype=np.float64)
    return np.stack([norm_fp16_ru_bits(vh, v), norm_fp16_ru_bits(v, np.zeros_like(v))], axis=-1)


def witness_bits(k_hat: np.ndarray, k32: np.ndarray) -> np.ndarray:
    """fp16 patterns of the band norms of r = k_hat - k (WitCert §4.1, eq. (2)): each the exact
    norm of the band's residual, rounded up."""
    kh = np.asarray(k_hat, dtype=np.float64)
    k = np.asarray(k32, dtype=np.float32).astype(np.float64)
    return norm_fp16_ru_bits(_band_view(kh), _band_view(k))
