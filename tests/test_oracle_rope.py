"""Pins of the oracle's binary32 RoPE-on-append (CPU).

* position 0 is the identity exactly (cos 1, sin 0);
* a closed form: the unit vector on channel j rotates to (fl(cos a), fl(sin a)) at pair j;
* each rotated channel is within one rounding of each of its three binary32 steps of the float64
  rotation with the same table, and pair norms are kept to that accuracy;
* the table and the rotation agree with the input generator's independently written float64 RoPE
  (angle formula, half-split pairing, sign convention) within the table's and the steps' rounding;
* a mistake in the pairing, the sign or the frequency breaks the last check by orders of magnitude.
"""
import numpy as np

import workloads as W
from oracle.rope import cos_sin_table, rope_fp32

U = 2.0 ** -24   # unit roundoff of binary32


def _keys(n, heads=1, seed=0):
    return (np.random.default_rng(seed).standard_normal((n, heads, 128)) * 3).astype(np.float32)


def test_position_zero_is_the_identity():
    t = cos_sin_table(8)
    assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)
    k = _keys(5, 4)
    assert np.array_equal(rope_fp32(k, np.zeros(5, dtype=np.int64), t), k)


def test_unit_vector_closed_form():
    theta, pos = 1e6, 7
    t = cos_sin_table(pos + 1, theta)
    for j in (0, 1, 17, 63):
        k = np.zeros((1, 128), dtype=np.float32)
        k[0, j] = 1.0
        r = rope_fp32(k, np.array([pos]), t)[0]
        a = pos * theta ** (-2.0 * j / 128)
        assert r[j] == np.float32(np.cos(a)) and r[j + 64] == np.float32(np.sin(a))
        assert np.count_nonzero(r) == 2


def test_within_one_rounding_per_step_of_the_float64_rotation():
    t = cos_sin_table(4096)
    pos = np.random.default_rng(1).integers(0, 4096, 300)
    k = _keys(300, 8, seed=2)
    r = rope_fp32(k, pos, t).astype(np.float64)
    c, s = t[pos, None, :64].astype(np.float64), t[pos, None, 64:].astype(np.float64)
    x, y = k[..., :64].astype(np.float64), k[..., 64:].astype(np.float64)
    ex, ey = x * c - y * s, y * c + x * s
    # fl(fl(xc) - fl(ys)): |error| <= u (|xc| + |ys|) + u |result| (plus the products' own rounding)
    bx = U * (np.abs(x * c) + np.abs(y * s)) * 1.0000001 + U * np.abs(ex) * 1.0000001
    by = U * (np.abs(y * c) + np.abs(x * s)) * 1.0000001 + U * np.abs(ey) * 1.0000001
    assert np.all(np.abs(r[..., :64] - ex) <= bx + 2.0 ** -149)
    assert np.all(np.abs(r[..., 64:] - ey) <= by + 2.0 ** -149)
    # pair norms are kept to the same accuracy (|cos^2 + sin^2 - 1| of the table is within 4u)
    n0 = np.hypot(x, y)
    n1 = np.hypot(r[..., :64], r[..., 64:])
    assert np.all(np.abs(n1 - n0) <= 8 * U * n0 + 2.0 ** -140)
    tt = t.astype(np.float64)
    assert np.max(np.abs(tt[:, :64] ** 2 + tt[:, 64:] ** 2 - 1.0)) <= 4 * U


def test_agrees_with_the_generators_float64_rope():
    theta = 1e6
    pos = np.random.default_rng(3).integers(0, 65536, 400)
    t = cos_sin_table(65536, theta)
    k = _keys(400, 4, seed=4)
    mine = rope_fp32(k, pos, t).astype(np.float64)
    ref = W.apply_rope(k, pos, theta).astype(np.float64)   # float64 math, rounded once
    scale = np.abs(k).astype(np.float64).max(axis=-1, keepdims=True)
    assert np.max(np.abs(mine - ref) / scale) <= 8 * U
    # the likely mistakes are caught: interleaved pairs (2j, 2j + 1) rotated instead of (j, j + 64), a
    # flipped sine, a wrong frequency
    gathered = np.concatenate([k[..., 0::2], k[..., 1::2]], axis=-1)     # pair (2j, 2j + 1) -> (j, j + 64)
    r = rope_fp32(gathered, pos, t)
    interleaved = np.empty_like(r)
    interleaved[..., 0::2], interleaved[..., 1::2] = r[..., :64], r[..., 64:]
    assert np.max(np.abs(interleaved - ref) / scale) > 1e-2
    flipped = t.copy()
    flipped[:, 64:] *= -1
    assert np.max(np.abs(rope_fp32(k, pos, flipped) - ref) / scale) > 1e-2
    assert np.max(np.abs(rope_fp32(k, pos, cos_sin_table(65536, 1e4)) - ref) / scale) > 1e-2
