"""Pins of the oracle's number encoders against independent conversions and closed forms (CPU)."""
import numpy as np
import pytest
import torch

from oracle.encoders import (
    bf16_bits_rne,
    bf16_value,
    e4m3_bits_rne_satfinite,
    e4m3_value,
    fp16_bits,
    fp16_value,
    round_to_grid,
)


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


def test_bf16_matches_torch_conversion():
    x = _random_f32(1 << 20, 1)
    # add exact ties and near-ties around 1.0
    base = np.float32(1.0).view(np.uint32)
    extra = np.array([base + d for d in (0x7FFF, 0x8000, 0x8001, 0x17FFF, 0x18000, 0x18001)], dtype=np.uint32).view(np.float32)
    x = np.concatenate([x, extra, np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], dtype=np.float32)])
    ours = bf16_bits_rne(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(bf16_value(ours[nan])))


def test_bf16_tie_cases_closed_form():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even significand (1.0)
    assert bf16_value(bf16_bits_rne(np.float32(1 + 2**-8)))[()] == 1.0
    assert bf16_value(bf16_bits_rne(np.float32(1 + 3 * 2**-8)))[()] == 1 + 2**-6
    assert bf16_value(bf16_bits_rne(np.float32(1 + 2**-8 + 2**-20)))[()] == 1 + 2**-7


@pytest.mark.parametrize("scale", [1.0, 2.0**-14, 2.0**-20, 6.0e4])
def test_fp16_rne_matches_numpy(scale):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200_000) * scale
    ours = fp16_bits(x, "rne")
    with np.errstate(over="ignore"):   # the 6e4 scale reaches past the fp16 range on purpose (-> inf)
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_ru_is_smallest_upper_bound():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.random(100_000) * 10, rng.random(10_000) * 2**-15, rng.random(1000) * 65504,
                        -rng.random(1000) * 3, np.array([0.0, 1.0, 65504.0, 2**-24, 3 * 2**-25])])
    h = fp16_bits(x, "ru")
    v = fp16_value(h)
    assert np.all(v >= x)
    below = np.nextafter(h.view(np.float16), np.float16(-np.inf)).astype(np.float64)
    assert np.all(below < x)
    # overflow past the largest finite value rounds up to +inf
    assert np.isinf(fp16_value(fp16_bits(np.array([65504.5]), "ru")))[0]
    assert fp16_value(fp16_bits(np.array([-70000.0]), "ru"))[0] == -65504.0
    # infinities convert to themselves in both modes (IEEE 754 conversion of an infinity)
    for mode in ("rne", "ru"):
        assert list(fp16_bits(np.array([np.inf, -np.inf]), mode)) == [0x7C00, 0xFC00]


def test_e4m3_decoder_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_value(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert e4m3_value(np.uint8(0x7E))[()] == 448.0


def test_e4m3_encoder_matches_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200_000) * s for s in (1.0, 100.0, 2**-7, 2**-10)]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ours = e4m3_bits_rne_satfinite(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturation_and_ties_closed_form():
    vals = np.array([449.0, 463.9, 464.0, 1e6, np.inf, -1e9, 2**-10, 3 * 2**-10, 2**-9 * 1.5], dtype=np.float32)
    out = e4m3_value(e4m3_bits_rne_satfinite(vals))
    # beyond 448 saturates; 2^-10 is half the smallest subnormal 2^-9: ties to even -> 0;
    # 3*2^-10 = 1.5 * 2^-9 ties to 2 * 2^-9; the last equals the same tie
    assert list(out) == [448.0, 448.0, 448.0, 448.0, 448.0, -448.0, 0.0, 2 * 2**-9, 2 * 2**-9]
    assert e4m3_bits_rne_satfinite(np.float32(np.nan))[()] == 0x7F


def test_round_to_grid_directed_modes_bracket():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(50_000) * 7
    up = round_to_grid(x, 10, -14, "ru")
    dn = round_to_grid(x, 10, -14, "rd")
    ne = round_to_grid(x, 10, -14, "rne")
    assert np.all(dn <= x) and np.all(x <= up)
    assert np.all((ne == up) | (ne == dn))
