"""Pins of the oracle's Philox4x32-10 stream and dither (CPU).

Agreement with an external Philox implementation is checked on the GPU (cuRAND's
Philox4x32-10, tests/test_gpu_philox_pin.py).  Here the generator is pinned by
properties that a plausible mistake (a wrong multiplier, a swapped word, a
missing key bump, a wrong output-word mapping) breaks:

* bijectivity: an independently written inverse recovers the counter;
* the inverse uses the key schedule and multipliers in the opposite order, so
  a round written with swapped output words fails it;
* uniformity, independence and avalanche statistics;
* the dither values lie on the documented 256-point grid, are exact in fp16,
  come from the documented bit fields of the documented words, and are
  uniform (chi-square) with the four fields of a word disjoint (together they
  rebuild the word) and pairwise independent;
* the subtractively dithered rounding error on that grid: its mean over the
  grid is within 2^-9 of 0 for every input (exhaustive over the grid), and
  its centred moment generating function stays below exp(l^2/24), the
  variance proxy 1/12 that Tier B uses.
"""
import numpy as np
import pytest

from oracle import philox as P


def _inv_mod_2_32(m):
    return pow(int(m), -1, 1 << 32)


def _philox_inverse(y, key, rounds=10):
    """Invert Philox4x32-``rounds`` written from the round definition (not from philox4x32_10)."""
    y0, y1, y2, y3 = (np.asarray(v, dtype=np.uint64) for v in y)
    mask = np.uint64(0xFFFFFFFF)
    keys = []
    k0, k1 = int(key[0]), int(key[1])
    for r in range(rounds):
        keys.append((k0, k1))
        k0 = (k0 + 0x9E3779B9) & 0xFFFFFFFF
        k1 = (k1 + 0xBB67AE85) & 0xFFFFFFFF
    inv0 = np.uint64(_inv_mod_2_32(0xD2511F53))
    inv1 = np.uint64(_inv_mod_2_32(0xCD9E8D57))
    for r in reversed(range(rounds)):
        kk0, kk1 = keys[r]
        # forward: y1 = lo(M1*x2), y3 = lo(M0*x0), y0 = hi(M1*x2)^x1^k0, y2 = hi(M0*x0)^x3^k1
        x2 = (y1 * inv1) & mask
        x0 = (y3 * inv0) & mask
        hi1 = (np.uint64(0xCD9E8D57) * x2) >> np.uint64(32)
        hi0 = (np.uint64(0xD2511F53) * x0) >> np.uint64(32)
        x1 = y0 ^ hi1 ^ np.uint64(kk0)
        x3 = y2 ^ hi0 ^ np.uint64(kk1)
        y0, y1, y2, y3 = x0, x1, x2, x3
    return y0, y1, y2, y3


def test_constants_are_the_published_ones():
    # Weyl constants: floor(2^32 * (golden ratio - 1)) and floor(2^32 * (sqrt(3) - 1))
    import math
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    phi = (1 + Decimal(5).sqrt()) / 2
    assert P.PHILOX_W0 == int((phi - 1) * (1 << 32))
    assert P.PHILOX_W1 == int((Decimal(3).sqrt() - 1) * (1 << 32))
    assert P.PHILOX_M0 % 2 == 1 and P.PHILOX_M1 % 2 == 1  # odd, hence invertible mod 2^32
    assert math.gcd(P.PHILOX_M0, 1 << 32) == 1


def test_bijective_via_independent_inverse():
    rng = np.random.default_rng(11)
    ctr = [rng.integers(0, 2**32, 10_000, dtype=np.uint64) for _ in range(4)]
    key = (0x1234ABCD, 0xDEADBEEF)
    y = P.philox4x32_10(ctr, key)
    back = _philox_inverse(y, key)
    for a, b in zip(ctr, back):
        assert np.array_equal(a, b)


def test_single_round_structure():
    # one round with key (0, 0) on counter (1, 0, 0, 0): only the first product is non-zero
    y = P.philox4x32_10(([1], [0], [0], [0]), (0, 0), rounds=1)
    assert [int(v[0]) for v in y] == [0, 0, 0, P.PHILOX_M0]
    y = P.philox4x32_10(([0], [0], [1], [0]), (0, 0), rounds=1)
    assert [int(v[0]) for v in y] == [0, P.PHILOX_M1, 0, 0]
    y = P.philox4x32_10(([0], [5], [0], [7]), (3, 9), rounds=1)
    assert [int(v[0]) for v in y] == [5 ^ 3, 0, 7 ^ 9, 0]


def test_uniform_and_independent_words():
    n = 1 << 18
    slots = np.arange(n, dtype=np.uint64)
    w = P.philox4x32_10((slots, np.uint64(3), np.uint64(1), np.uint64(7)), (42, 0))
    allw = np.concatenate([v for v in w]).astype(np.float64) / 2**32
    # chi-square on 256 bins
    hist = np.bincount((allw * 256).astype(int), minlength=256)
    exp = allw.size / 256
    chi2 = np.sum((hist - exp) ** 2 / exp)
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    # words of one call are uncorrelated
    c = np.corrcoef(np.stack([v.astype(np.float64) for v in w]))
    assert np.max(np.abs(c - np.eye(4))) < 0.01


def test_avalanche():
    rng = np.random.default_rng(12)
    ctr = [rng.integers(0, 2**32, 4096, dtype=np.uint64) for _ in range(4)]
    base = P.philox4x32_10(ctr, (7, 8))
    flipped = [c.copy() for c in ctr]
    flipped[2] ^= np.uint64(1 << 13)
    out = P.philox4x32_10(flipped, (7, 8))
    diff = sum(np.unpackbits((a ^ b).astype(np.uint32).view(np.uint8)).sum() for a, b in zip(base, out))
    frac = diff / (4096 * 128)
    assert abs(frac - 0.5) < 0.01


def test_dither_grid_range_and_moments():
    slots = np.arange(20_000)[:, None]
    ch = np.arange(128)[None, :]
    xi = P.dither(0xABCDEF0123, layer=5, kv_head=2, slot=slots, channel=ch)
    assert xi.shape == (20_000, 128)
    assert np.all(xi >= -0.5) and np.all(xi < 0.5)
    n = (xi + 0.5) * 256
    assert np.array_equal(n, np.round(n))                        # on the 2^-8 grid
    assert np.all(np.float16(xi).astype(np.float64) == xi)       # exact in fp16
    # xi + 9/2 is the fp16 number 4 + field / 256: its bit pattern is 0x4400 | field (-(xi + 9/2): 0xC400 | field)
    f = P.dither_fields(0xABCDEF0123, 5, 2, slots, ch)
    assert np.array_equal(np.float16(xi + 4.5).view(np.uint16).astype(np.uint64), np.uint64(0x4400) | f)
    assert np.array_equal(np.float16(-(xi + 4.5)).view(np.uint16).astype(np.uint64), np.uint64(0xC400) | f)
    # grid mean -2^-9, variance (1 - 2^-16) / 12
    assert abs(xi.mean() + 2**-9) < 3 * np.sqrt(1 / 12 / xi.size)
    assert abs(xi.var() - (1 - 2**-16) / 12) < 0.002
    counts = np.bincount(n.astype(np.int64).ravel(), minlength=256)
    expect = xi.size / 256
    chi2 = float(np.sum((counts - expect) ** 2 / expect))
    assert chi2 < 255 + 5 * np.sqrt(2 * 255)                    # ~5 sigma of chi-square(255)


def test_dither_fields_of_one_word_are_disjoint_and_independent():
    slots = np.arange(200_000)
    w = P.dither_words(17, 3, 1, slots, 12)                       # word 3 of the call: channels 12..15
    fields = [P.dither_fields(17, 3, 1, slots, c) for c in (12, 13, 14, 15)]
    # the fields are the word's bytes, lowest first: via the little-endian byte view of the words
    as_bytes = w.astype(np.uint32).astype("<u4").view(np.uint8).reshape(-1, 4)
    for i in range(4):
        assert np.array_equal(fields[i], as_bytes[:, i].astype(np.uint64))
    # the four fields are 32 disjoint bits of the word: together they rebuild it
    back = fields[0] + fields[1] * np.uint64(256) + fields[2] * np.uint64(65536) + fields[3] * np.uint64(16777216)
    assert np.array_equal(back, w)
    for i in range(4):
        for j in range(i + 1, 4):
            a, b = fields[i], fields[j]
            joint = np.bincount(((a >> np.uint64(3)) * np.uint64(32) + (b >> np.uint64(3))).astype(np.int64),
                                minlength=1024)
            expect = slots.size / 1024
            chi2 = float(np.sum((joint - expect) ** 2 / expect))
            assert chi2 < 1023 + 5 * np.sqrt(2 * 1023)
            assert abs(np.corrcoef(a.astype(np.float64), b.astype(np.float64))[0, 1]) < 0.01


N_GRID = 1 << P.DITHER_BITS


def _grid_errors(y):
    """rint(fp32(y + xi)) - (y + xi) for every xi of the grid (float64, exact), y [..] fp32 -> [.., 256]."""
    xi = np.arange(N_GRID) * 2.0**-8 - 0.5
    y = np.asarray(y, dtype=np.float32).astype(np.float64)[..., None]
    y2 = (y + xi).astype(np.float32).astype(np.float64)
    return np.rint(y2) - (y + xi)


def test_subtractive_error_bias_exhaustive_over_the_grid():
    rng = np.random.default_rng(5)
    ys = np.concatenate([
        rng.uniform(-126.5, 126.5, 4000),
        np.arange(-126.5, 127.0, 0.5),                            # half-integers and integers
        np.arange(-4, 4, 2.0**-12),                               # inputs on and off the dither grid
        np.array([0.0, 2.0**-30, -2.0**-30, 126.5, -126.5, 0.5 - 2.0**-9, 0.25 + 2.0**-11]),
    ]).astype(np.float32)
    e = _grid_errors(ys)
    # subtractive dither: |error| <= 1/2 LSB, up to the binary32 rounding of y + xi
    assert np.all(np.abs(e) <= 0.5 + 2.0**-24)
    mu = e.mean(axis=-1)
    bound = P.subtractive_error_bias_bound()
    assert bound == 2.0**-9
    assert np.max(np.abs(mu)) <= bound * (1 + 1e-9) + 2.0**-24   # within half a grid step
    assert np.max(np.abs(mu)) > 0.9 * bound                      # and the bound is reached: the grid does bias
    # the errors are the grid itself, shifted: sorted, consecutive gaps of 2^-8
    gaps = np.diff(np.sort(e[: 4000], axis=-1), axis=-1)
    assert np.allclose(gaps, 2.0**-8, rtol=0, atol=2.0**-20)


def test_subtractive_error_centred_mgf_proxy():
    rng = np.random.default_rng(6)
    e = _grid_errors(rng.uniform(-126.5, 126.5, 500).astype(np.float32))
    c = e - e.mean(axis=-1, keepdims=True)
    for lam in (0.1, 1.0, 3.0, 8.0, 20.0):
        mgf = np.exp(lam * c).mean(axis=-1)
        assert np.all(mgf <= np.exp(lam * lam / 24) * (1 + 1e-12))
        # and equals the closed form of the centred N-point grid, sinh(l/2) / (N sinh(l / 2N))
        closed = np.sinh(lam / 2) / (N_GRID * np.sinh(lam / (2 * N_GRID)))
        assert np.allclose(mgf, closed, rtol=1e-9)


def test_dither_stream_is_keyed_by_every_coordinate():
    base = P.dither(99, 1, 0, np.arange(1000), 0)
    assert not np.array_equal(base, P.dither(100, 1, 0, np.arange(1000), 0))   # seed
    assert not np.array_equal(base, P.dither(99, 2, 0, np.arange(1000), 0))   # layer
    assert not np.array_equal(base, P.dither(99, 1, 1, np.arange(1000), 0))   # kv head
    assert not np.array_equal(base, P.dither(99, 1, 0, np.arange(1, 1001), 0))  # slot
    # the sixteen channels of one call: channel c <- byte c & 3 of word c >> 2
    w = P.philox4x32_10((np.arange(5, dtype=np.uint64), np.uint64(1), np.uint64(0), np.uint64(0)), (99, 0))
    for c in range(16):
        xi = P.dither(99, 1, 0, np.arange(5), c)
        field = (w[c >> 2] // np.uint64(256 ** (c & 3))) % np.uint64(256)
        assert np.array_equal(xi, field.astype(np.float64) / 256 - 0.5)
    # channel 16 starts the next call
    w1 = P.philox4x32_10((np.arange(5, dtype=np.uint64), np.uint64(1), np.uint64(0), np.uint64(1)), (99, 0))
    assert np.array_equal(P.dither(99, 1, 0, np.arange(5), 16),
                          (w1[0] % np.uint64(256)).astype(np.float64) / 256 - 0.5)
    # stream uniqueness: distinct (slot, layer, head, channel-group) tuples give distinct words
    slots = np.repeat(np.arange(64), 32 * 2)
    heads = np.tile(np.repeat(np.arange(2), 32), 64)
    groups = np.tile(np.arange(32), 128)   # (16 calls per row; any 32 distinct groups serve the check)
    words = P.philox4x32_10((slots.astype(np.uint64), np.uint64(3), heads.astype(np.uint64), groups.astype(np.uint64)), (5, 6))
    packed = set(zip(*(v.tolist() for v in words)))
    assert len(packed) == slots.size
