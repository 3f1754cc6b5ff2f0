"""Number-format encoders, written from the format definitions (oracle; test infrastructure).

Formats (IEEE 754 binary16; bfloat16 = the top 16 bits of binary32; OCP FP8
E4M3 "fn": 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities, the
all-ones pattern S.1111.111 is NaN, largest finite 448).

The layouts come from "Compress the shared cartridge" (K16/V8: BF16 keys, FP8
E4M3 values; K8/V8: E4M3 keys too).  The rounding modes come from "WitCert"
§4.1 eq. (2) (the witness is stored in fp16, rounded *up* so that it never
under-states the residual norm) and §6.2.1 (quantize with the stored fp16
scale, round-to-nearest).

Every encoder here works on exact dyadic values in float64: a value is split
into (integer significand, power-of-two ulp) for its binade and the significand
is rounded with the requested mode.  Nothing is borrowed from a library
conversion routine; the tests pin these functions against numpy / torch's own
conversions and against closed forms.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_grid",
    "f32",
    "bf16_bits_rne",
    "bf16_value",
    "fp16_bits",
    "fp16_value",
    "e4m3_bits_rne_satfinite",
    "e4m3_value",
]


def f32(x) -> np.ndarray:
    """Round float64 values to binary32 (round-to-nearest-even).

    Each oracle step that the CUDA path performs in fp32 is evaluated here in
    float64 and rounded once with this function.  For + - * / and sqrt of
    binary32 operands that double rounding equals the correctly rounded binary32
    result, because 53 >= 2*24 + 2.
    """
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_to_grid(x: np.ndarray, mant_bits: int, emin: int, mode: str) -> np.ndarray:
    """Round float64 ``x`` to a binary floating-point grid with unlimited exponent range above.

    ``mant_bits`` fraction bits, smallest normal exponent ``emin`` (values below
    2**emin are on the subnormal grid with spacing 2**(emin - mant_bits)).
    ``mode``: 'rne' (nearest, ties to even), 'ru' (toward +inf), 'rd' (toward -inf).
    Returns float64 values exactly on the grid.  Overflow is handled by callers.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    finite = np.isfinite(x)
    nz = finite & (x != 0)
    ax = np.abs(x[nz])
    # exponent of the binade: ax in [2**e, 2**(e+1)); np.frexp gives ax = m * 2**k, m in [0.5, 1)
    _, k = np.frexp(ax)
    e = np.maximum(k.astype(np.int64) - 1, emin)
    ulp = np.ldexp(1.0, (e - mant_bits).astype(np.int64))
    q = ax / ulp  # exact: division by a power of two
    neg = x[nz] < 0
    if mode == "rne":
        n = np.rint(q)  # numpy rint is round-half-to-even
    elif mode == "ru":
        # toward +inf: magnitude rounds up for positives, down for negatives
        n = np.where(neg, np.floor(q), np.ceil(q))
    elif mode == "rd":
        n = np.where(neg, np.ceil(q), np.floor(q))
    else:
        raise ValueError(mode)
    val = n * ulp  # exact (n has at most mant_bits+1 bits, or is 2**(mant_bits+1))
    out[nz] = np.where(neg, -val, val)
    out[~finite] = x[~finite]
    # keep the sign of zero results (irrelevant for the encoders below, which work on magnitudes)
    return out


# ----------------------------------------------------------------------------- bfloat16

def bf16_bits_rne(x32: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bit patterns, round-to-nearest-even (NaN -> quiet NaN 0x7FC0 | sign).

    bfloat16 keeps binary32's 8-bit exponent and 7 fraction bits, so its grid
    is binary32's with 16 fewer fraction bits, including the subnormals.
    """
    with np.errstate(invalid="ignore"):
        x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    r = round_to_grid(x, 7, -126, "rne")
    sign = np.signbit(x)
    # overflow: values that round above the largest finite bf16 become inf
    big = np.abs(r) > float.fromhex("0x1.fep127")  # largest finite bfloat16: (2 - 2**-7) * 2**127
    r = np.where(big, np.where(sign, -np.inf, np.inf), r)
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    # a zero result keeps the input's sign (bf16 of -tiny is -0)
    bits = np.where((r == 0) & sign, np.uint16(0x8000), bits)
    bits = np.where(np.isnan(x), np.where(sign, np.uint16(0xFFC0), np.uint16(0x7FC0)), bits)
    return bits.astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- binary16

_FP16_MAX = 65504.0


def fp16_bits(x: np.ndarray, mode: str = "rne") -> np.ndarray:
    """float64 -> IEEE binary16 bit patterns with rounding ``mode`` ('rne' or 'ru').

    10 fraction bits, smallest normal 2**-14, subnormal spacing 2**-24.
    Overflow follows IEEE: round-to-nearest overflows to inf at or above
    65520 (the midpoint past 65504); round-up overflows to inf above 65504
    (and a finite negative value never rounds up to -inf); an infinity converts
    to the infinity of its sign in either mode.
    """
    x = np.asarray(x, dtype=np.float64)
    r = round_to_grid(x, 10, -14, mode)
    sign = np.signbit(x)
    if mode == "rne":
        over = np.abs(r) > _FP16_MAX
        r = np.where(over, np.where(sign, -np.inf, np.inf), r)
    elif mode == "ru":
        r = np.where(r > _FP16_MAX, np.inf, r)
        # a finite value below -65504 rounds up to -65504; -inf itself converts to -inf
        r = np.where((r < -_FP16_MAX) & np.isfinite(r), -_FP16_MAX, r)
    else:
        raise ValueError(mode)
    # r is exactly representable in binary16 (or +-inf/nan): the numpy cast of an
    # exactly representable value is exact, so it only builds the bit pattern.
    h = r.astype(np.float16).view(np.uint16)
    h = np.where((r == 0) & sign, np.uint16(0x8000), h)
    h = np.where(np.isnan(x), np.uint16(0x7E00), h)
    return h.astype(np.uint16)


def fp16_value(bits: np.ndarray) -> np.ndarray:
    """binary16 bit patterns -> float64 values (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ----------------------------------------------------------------------------- FP8 E4M3

E4M3_MAX = 448.0


def e4m3_bits_rne_satfinite(x32: np.ndarray) -> np.ndarray:
    """binary32 -> FP8 E4M3 bit patterns: round-to-nearest-even, saturate to +-448, NaN -> 0x7F.

    E4M3: exponent bias 7, 3 fraction bits, normals 2**-6 .. 448, subnormals
    k * 2**-9.  "satfinite": a finite value whose rounded magnitude exceeds
    448 (and +-inf) becomes +-448.  The sign of zero is kept.
    """
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    ax = np.abs(x)
    r = round_to_grid(np.where(np.isinf(ax), E4M3_MAX, ax), 3, -6, "rne")
    r = np.minimum(r, E4M3_MAX)
    # encode the magnitude
    bits = np.zeros(x.shape, dtype=np.uint16)
    sub = r < 2.0 ** -6
    # subnormal: value = m * 2**-9, m in 0..7, exponent field 0
    rr = np.where(np.isnan(r), 0.0, r)  # NaN inputs are patched below
    m_sub = np.rint(rr * 2.0 ** 9).astype(np.int64)
    # normal: value = (1 + f/8) * 2**e, field = e + 7
    _, k = np.frexp(np.where(sub, 1.0, rr))
    e = k.astype(np.int64) - 1
    f = np.rint((np.where(sub, 1.0, rr) / np.ldexp(1.0, e) - 1.0) * 8).astype(np.int64)
    norm_bits = ((e + 7) << 3) | f
    bits = np.where(sub, m_sub, norm_bits).astype(np.uint16)
    bits = bits | np.where(sign, np.uint16(0x80), np.uint16(0)).astype(np.uint16)
    bits = np.where(np.isnan(x), np.where(sign, np.uint16(0xFF), np.uint16(0x7F)), bits)
    return bits.astype(np.uint8)


def e4m3_value(bits: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bit patterns -> float64 values (NaN for S.1111.111)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    ef = (b >> 3) & 0xF
    f = b & 0x7
    val = np.where(ef == 0, f * 2.0 ** -9, (1.0 + f / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((ef == 15) & (f == 7), np.nan, val)
    return s * val
