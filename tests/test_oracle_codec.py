"""Pins of the oracle's E4M3 / BF16 codecs and of the ExpCast byte mapping.

Each test checks the oracle against something other than itself: torch's
float8_e4m3fn conversions (an independent library routine), the format
definition, and the numbers the VC-Attention summary prints in its
"ExpCast-FP8" section (tests/golden/expcast_facts.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "expcast_facts.json")))


def test_decode_table_matches_torch_float8():
    tab = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(tab[~nan], ref[~nan])
    assert tab[0x7E] == 448.0 and tab[1] == 2.0 ** -9 and tab[8] == 2.0 ** -6


def _torch_cast(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    mags = 2.0 ** rng.uniform(-12, np.log2(448.0), 4000)
    x = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    assert np.array_equal(oracle.e4m3_encode_array(x), _torch_cast(x))


def test_encode_ties_to_even_and_midpoints():
    tab = oracle.e4m3_table()
    codes = np.arange(0, 126)
    mids = ((tab[codes] + tab[codes + 1]) / 2).astype(np.float32)   # exact in float32
    got = oracle.e4m3_encode_array(mids)
    even = np.where(codes % 2 == 0, codes, codes + 1)
    assert np.array_equal(got, even.astype(np.uint8))
    assert np.array_equal(got, _torch_cast(mids))


def test_encode_decode_roundtrip_and_saturation():
    tab = oracle.e4m3_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_from_float(tab[c]) == c
    assert oracle.e4m3_from_float(448.0) == 0x7E
    assert oracle.e4m3_from_float(1e9) == 0x7E
    assert oracle.e4m3_from_float(-470.0) == 0xFE
    assert oracle.e4m3_from_float(2.0 ** -11) == 0      # below half the smallest subnormal
    assert oracle.e4m3_from_float(float("nan")) == 0x7F


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(3000) * 10.0 ** rng.uniform(-5, 5, 3000)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_from_double(x), ref)


def test_byte_relation_over_all_normal_codes():
    """An E4M3 code read as an integer is 8*log2(value)+56, up to the mantissa
    curvature, for every normal code; subnormals, zero and NaN are exceptions."""
    g = GOLDEN["byte_relation"]
    tab = oracle.e4m3_table()
    for c in range(8, 127):
        dev = c - (g["slope"] * math.log2(tab[c]) + g["offset"])
        assert -0.6800 <= dev <= 1e-12, (c, dev)
        neg = (c | 0x80)
        assert tab[neg] == -tab[c]
    worst = min(c - (8 * math.log2(tab[c]) + 56) for c in range(8, 127))
    # code 8e+m is worth 2^(e-7)(1+m/8): deviation m - 8 log2(1+m/8), worst at m = 4
    assert worst == pytest.approx(4 - 8 * math.log2(1.5), abs=1e-12)
    bad = [c for c in range(1, 8) if not (-0.68 <= c - (8 * math.log2(tab[c]) + 56) <= 0)]
    assert bad == list(range(1, 8))


def _expcast_vs_cast(L):
    """ExpCast byte and exp-then-cast byte for stored values v = 2^L.

    With c0 = 120 a score Z (code units) relative to reference 0 stores
    v = 2^(Z/8 + 8), so Z = 8 L - 64."""
    direct = oracle.expcast_codes(8.0 * L - 64.0, 0.0)
    cast = oracle.e4m3_encode_array(np.exp2(L))
    return direct.astype(int), cast.astype(int)


def test_expcast_match_rate_and_distance():
    g = GOLDEN["match_rate"]
    rng = np.random.default_rng(3)
    L = rng.uniform(-6.0, math.log2(448.0) - 0.2, 200_000)
    direct, cast = _expcast_vs_cast(L)
    rate = float(np.mean(direct == cast))
    assert abs(rate - g["value"]) < 0.003, rate
    assert int(np.max(np.abs(direct - cast))) == g["max_code_distance"]


def test_expcast_rounding_mode_is_nearest_not_floor():
    """Truncating the FMA result instead of rounding it would give ~61 %."""
    rng = np.random.default_rng(4)
    L = rng.uniform(-6.0, math.log2(448.0) - 0.2, 50_000)
    cast = oracle.e4m3_encode_array(np.exp2(L)).astype(int)
    trunc = np.floor(8 * L + 56 + GOLDEN["beta"]["value"]).astype(int)
    assert np.mean(trunc == cast) < 0.65
    direct, _ = _expcast_vs_cast(L)
    assert np.mean(direct == cast) > 0.79


def test_expcast_total_variation_bound():
    """Worst-case ratio dec(code(v))/v over the normal range fixes the TV bound."""
    g = GOLDEN["tv_bound"]
    L = np.linspace(-5.9, 8.0, 400_001)
    codes = oracle.expcast_codes(8.0 * L - 64.0, 0.0)
    tab = oracle.e4m3_table()
    ratio = tab[codes] / np.exp2(L)
    R = ratio.max() / ratio.min()
    tv = (math.sqrt(R) - 1) / (math.sqrt(R) + 1)
    assert tv < g["value"]
    assert tv == pytest.approx(0.03637, abs=2e-4)


def test_expcast_row_total_variation_on_random_rows():
    g = GOLDEN["tv_bound"]
    rng = np.random.default_rng(5)
    tab = oracle.e4m3_table()
    for _ in range(20):
        z = rng.standard_normal(512) * 3.0         # log2-domain scores
        Z = 8.0 * z
        m8 = np.ceil(Z.max() - 0.65) + 0.65
        codes = oracle.expcast_codes(Z, m8)
        p_hat = tab[codes]
        p = np.exp2((Z - m8) / 8.0)
        tv = 0.5 * np.abs(p_hat / p_hat.sum() - p / p.sum()).sum()
        underflow = p[codes == 0].sum() / p.sum()
        assert tv <= g["value"] + underflow + 1e-12


def test_expcast_clamps():
    assert oracle.expcast_code(-1e6, 0.0) == 0
    assert oracle.expcast_code(1e3, 0.0) == 126
    assert oracle.expcast_code(0.0, 0.0) == 120      # rint(119.65)


@pytest.mark.parametrize("beta,c0", [(0.0, 120.0), (-0.35, 119.0), (-0.85, 120.0)])
def test_match_rate_pin_detects_wrong_constants(beta, c0):
    """The 79.6 % agreement fixes beta and c0: a shifted constant misses it."""
    rng = np.random.default_rng(6)
    L = rng.uniform(-6.0, math.log2(448.0) - 0.2, 40_000)
    direct = oracle.expcast_codes(8.0 * L - 64.0, 0.0, c0=c0, beta=beta).astype(int)
    cast = oracle.e4m3_encode_array(np.exp2(L)).astype(int)
    assert abs(np.mean(direct == cast) - GOLDEN["match_rate"]["value"]) > 0.01
