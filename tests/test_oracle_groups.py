"""CPU pins of the oracle's per-token channel-group scales (WitCert §6.2.3, Table 4; G_c = 32 by default).

* Table 4's byte account: K+V bytes per token per kv head and the saving against fp16 K+V for the block
  scale and the 16-, 32- and 128-channel token scales, and §6.2.3's 136 B per side (golden fixture).
* A hand-worked row: group scales, codes (round half to even, the dither added first) and the all-zero group.
* Locality: a channel changes only its own group's scale and codes; contiguous groups of G_c channels.
* Reductions: one group of 128 channels is the plain per-token INT8 quantizer, bit for bit, and its Tier B
  radius is the per-token radius; equal group scales give the per-token radius with that scale.
* Element bound |x_hat - x| <= s_g / 2 with the group's own scale (no code clips).
* Table 4's ordering of the paging-safe token granularities on keys with massive channels:
  16-channel groups <= 32-channel groups < one scalar per token (relative reconstruction error).
* Tier B with group scales: zero violations of |eps_t| <= u_t over dither seeds, and the variance
  proxy sum_c q_c^2 s_{g(c)}^2 / 12 matches the empirical variance of eps over dither seeds (so a
  radius built from the largest or the mean scale fails one side or the other).
"""
import json
import math
import os

import numpy as np

from oracle import attention as A
from oracle.bytes import int8_side_bytes, scale_granularity_saving
from oracle.encoders import fp16_value
from oracle.philox import dither
from oracle.quant import dequantize, dequantize_int8_groups, quantize, quantize_int8_groups
from workloads import apply_rope

SM = 1.0 / math.sqrt(128)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scale_granularity.json")


def _xi(seed, S, layer=0, head=0):
    return dither(seed, layer, head, np.arange(S)[:, None], np.arange(128)[None, :])


def _massive_keys(S, seed, channels=(3, 40, 71, 100), massive=40.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, 128))
    k[:, list(channels)] *= massive
    return apply_rope(k, np.arange(S))


def test_table4_byte_account():
    with open(GOLDEN) as f:
        g = json.load(f)
    assert 2 * 2 * g["head_dim"] == g["fp16_k_plus_v_bytes"]
    for row in g["rows"]:
        if row["granularity"] == "block":
            side = int8_side_bytes("block", block=row["block"])
        else:
            side = int8_side_bytes("token", group=row["group"])
        assert 2 * side == row["k_plus_v_bytes"], row["scheme"]
        assert round(100 * scale_granularity_saving(2 * side), 1) == row["saved_pct"], row["scheme"]
    assert int8_side_bytes("token", group=g["default_group"]) == g["bytes_per_side_default"]


def test_hand_worked_row():
    x = np.zeros(128, dtype=np.float32)
    xi = np.zeros(128)
    # group 0: amax 126.5 -> s = 1; ties go to even; the dither is added before rounding
    x[0], x[1], x[2], x[3], x[4], xi[4] = 126.5, 1.5, 2.5, -3.5, 0.25, 0.375
    # group 1: amax 253 -> s = 2
    x[32], x[33], x[34] = -253.0, 5.0, 7.0
    # group 2: all zero -> s = 0 and zero codes, even with a dither
    xi[64:96] = 0.4375
    # group 3: amax 1 -> s = fp16_rn(fp32(1 / 126.5)) = 2^-7 (1 + 12 / 1024) = 0x200C
    x[96], x[97], x[98] = 1.0, -0.5, 2.0 ** -30
    codes, sb, valid = quantize_int8_groups(x[None], xi[None], group=32)
    assert valid[0]
    assert sb[0].tolist() == [0x3C00, 0x4000, 0x0000, 0x200C]
    c = codes[0]
    assert c[:5].tolist() == [126, 2, 2, -4, 1]
    assert c[32:35].tolist() == [-126, 2, 4]     # -253/2 = -126.5 -> -126; 2.5 -> 2; 3.5 -> 4
    assert np.all(c[64:96] == 0)
    assert c[96:99].tolist() == [127, -63, 0]    # 1 / 0.0079040527 = 126.52 -> 127; -63.26 -> -63
    nz = np.zeros(128, dtype=bool)
    nz[[0, 1, 2, 3, 4, 32, 33, 34, 96, 97]] = True
    assert np.all(c[~nz] == 0)
    xh = dequantize_int8_groups(codes, sb, xi[None])[0]
    assert xh[0] == 126.0 and xh[4] == 1 - 0.375 and xh[32] == -252.0 and xh[96] == 127 * fp16_value(np.uint16(0x200C))


def test_groups_are_contiguous_and_local():
    k32 = _massive_keys(16, 1).astype(np.float32)
    xi = _xi(2, 16)
    c0, s0, _ = quantize_int8_groups(k32, xi, group=32)
    for ch in (0, 31, 32, 77, 127):
        k1 = k32.copy()
        k1[:, ch] = 500.0
        c1, s1, _ = quantize_int8_groups(k1, xi, group=32)
        g = ch // 32
        other = np.arange(4) != g
        assert np.array_equal(s1[:, other], s0[:, other]) and np.all(s1[:, g] != s0[:, g])
        keep = np.arange(128) // 32 != g
        assert np.array_equal(c1[:, keep], c0[:, keep])


def test_one_group_is_the_per_token_quantizer():
    k32 = _massive_keys(50, 3)
    xi = _xi(4, 50)
    c0, s0, v0 = quantize(k32, "int8", xi)
    c1, s1, v1 = quantize_int8_groups(k32, xi, group=128)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1[:, 0]) and np.array_equal(v0, v1)
    assert np.array_equal(dequantize(c0, s0, "int8", xi), dequantize_int8_groups(c1, s1, xi))
    q = np.random.default_rng(5).standard_normal(128)
    u0 = A.tier_b_radius(q, fp16_value(s0), SM, 50, 1e-2, 28, 28, 256)
    u1 = A.tier_b_radius_groups(q, fp16_value(s1), SM, 50, 1e-2, 28, 28, 256)
    assert np.allclose(u0, u1, rtol=1e-14, atol=0)
    # equal scales over four groups: the per-token radius with that scale
    s_eq = np.repeat(fp16_value(s0)[:, None], 4, axis=1)
    assert np.allclose(A.tier_b_radius_groups(q, s_eq, SM, 50, 1e-2, 28, 28, 256), u0, rtol=1e-14, atol=0)


def test_element_bound_with_the_groups_own_scale():
    k32 = _massive_keys(256, 6, massive=300.0)
    xi = _xi(7, 256)
    for group in (16, 32, 64):
        codes, sb, valid = quantize_int8_groups(k32, xi, group=group)
        assert np.all(valid) and np.all(np.abs(codes.astype(int)) <= 127)
        r = np.abs(dequantize_int8_groups(codes, sb, xi) - k32.astype(np.float64))
        s = np.repeat(fp16_value(sb), group, axis=1)
        assert np.all(r <= s / 2 * (1 + 1e-12))


def test_table4_ordering_of_token_granularities():
    k32 = _massive_keys(512, 8)
    xi = _xi(9, 512)
    err = {}
    for group in (16, 32, 128):
        codes, sb, _ = quantize_int8_groups(k32, xi, group=group)
        r = dequantize_int8_groups(codes, sb, xi) - k32.astype(np.float64)
        err[group] = np.linalg.norm(r) / np.linalg.norm(k32.astype(np.float64))
    assert err[16] <= err[32] < err[128]
    assert err[32] < 0.75 * err[128]


def _group_scales(S, seed):
    """Keys whose four groups have very different scales (massive channels in two groups only)."""
    return _massive_keys(S, seed, channels=(5, 6, 70), massive=30.0)


def test_tier_b_with_group_scales_zero_violations():
    S, H, L, T, dreq = 200, 4, 28, 256, 1e-2
    k32 = _group_scales(S, 10)
    q = np.random.default_rng(11).standard_normal((H, 128))
    viol = 0
    for seed in range(40):
        xi = _xi(2000 + seed, S)
        codes, sb, _ = quantize_int8_groups(k32, xi)
        kh = dequantize_int8_groups(codes, sb, xi)
        for h in range(H):
            eps = SM * (q[h] @ (kh - k32.astype(np.float64)).T)
            viol += int(np.sum(np.abs(eps) > A.tier_b_radius_groups(q[h], fp16_value(sb), SM, S, dreq, L, H, T)))
    assert viol == 0


def test_group_variance_proxy_matches_the_dither():
    S, n_seeds = 32, 600
    k32 = _group_scales(S, 12)
    q = np.random.default_rng(13).standard_normal(128)
    eps = np.empty((n_seeds, S))
    s_ref = None
    for seed in range(n_seeds):
        xi = _xi(5000 + seed, S)
        codes, sb, _ = quantize_int8_groups(k32, xi)
        s_ref = fp16_value(sb) if s_ref is None else s_ref
        assert np.array_equal(fp16_value(sb), s_ref)          # the scales do not depend on the dither
        eps[seed] = SM * (q @ (dequantize_int8_groups(codes, sb, xi) - k32.astype(np.float64)).T)
    qg2 = np.sum(q.reshape(4, 32) ** 2, axis=1)
    proxy = SM * SM * (s_ref ** 2 @ qg2) / 12                # per token
    ratio = eps.var(axis=0) / proxy
    # pooled over tokens: 32 x 600 draws, standard error of the mean ratio ~ 1 %
    assert abs(ratio.mean() - 1) < 0.04
    # the radius from the largest group scale over-states, the mean group scale under-states the spread
    big = SM * SM * np.sum(q ** 2) * s_ref.max(axis=1) ** 2 / 12
    mean = SM * SM * np.sum(q ** 2) * s_ref.mean(axis=1) ** 2 / 12
    assert np.mean(eps.var(axis=0) / big) < 0.5 and np.mean(eps.var(axis=0) / mean) > 1.3
    # the radius function's own sigma: u(S1) - u(S2) = (kappa1 - kappa2) sqrt(12 proxy) (the bias term cancels)
    d, L, H, T = 1e-2, 28, 28, 256
    kap = [math.sqrt(2.0 * math.log(2.0 * n / (d / (L * H * T))) / 12.0) for n in (100, 100000)]
    u1, u2 = (A.tier_b_radius_groups(q, s_ref, SM, n, d, L, H, T) for n in (100, 100000))
    sigma_fn = (u2 - u1) / (kap[1] - kap[0]) / math.sqrt(12.0)
    assert abs(np.mean(eps.var(axis=0) / sigma_fn ** 2) - 1) < 0.04
    # the mean error per token is within the grid's bias bound
    bias = SM * 2.0 ** -9 * (s_ref @ np.sum(np.abs(q.reshape(4, 32)), axis=1))
    assert np.all(np.abs(eps.mean(axis=0)) <= bias + 4 * np.sqrt(proxy / n_seeds))
