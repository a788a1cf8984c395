"""Pins of the oracle's baseline path: exp-then-cast probability bytes and the
natural key order, the standard FP8 kernel that ExpCast and the mid-window
order improve on ("Open-VC attention" news item, "Problem": one exponent per
score, then a conversion to FP8; "Architectural optimisations").

* The exp-then-cast byte equals torch's own float32 -> float8_e4m3fn cast of
  the stored value 2^((Z - m8 + c0 - 56)/8) (an independent implementation
  of the format's rounding).
* Against ExpCast it reproduces the agreement the VC-Attention summary
  reports ("ExpCast-FP8": the same byte on 79.6% of entries, otherwise one
  code away).
* Every output row lies within the rounding bound of E4M3 (relative error at
  most 2^-4 per normal probability) of exact attention on the same quantised
  inputs, plus the underflow tail.
* With the natural order the first visited block is block 0.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_attention import GOLDEN, SM, _bits, _exact_on_quantised, _inputs


def _torch_cast_codes(Z, m8):
    v = np.exp2((np.asarray(Z, np.float64) - m8 + oracle.C0 - 56.0) / 8.0)
    t = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("m8", [0.0, 17.65, -233.35])
def test_exp_cast_code_equals_torch_float8_cast(m8):
    rng = np.random.default_rng(7)
    # stored values from below the subnormal range up to 2^8.75
    Z = m8 + rng.uniform(-170.0, 6.0, 20_000)
    got = oracle.exp_cast_codes(Z, m8)
    want = _torch_cast_codes(Z, m8)
    assert np.array_equal(got, want)
    assert got.max() <= 126 and (got == 0).any()


def test_exp_cast_code_ties_and_edges():
    # v exactly on a code: 2^8 (p = 1) is code 120; 2^-9 (smallest subnormal) is code 1
    assert oracle.exp_cast_code(0.0) == 120
    assert oracle.exp_cast_code(8.0 * (-9 - 8)) == 1
    # half the smallest subnormal rounds to even (0); just above it rounds up
    assert oracle.exp_cast_code(8.0 * (-10 - 8)) == 0
    assert oracle.exp_cast_code(8.0 * (-10 - 8) + 1e-3) == 1


def test_exp_cast_agrees_with_expcast_as_reported():
    g = GOLDEN["match_rate"]
    rng = np.random.default_rng(3)
    L = rng.uniform(-6.0, math.log2(448.0) - 0.2, 100_000)    # normal range
    Z = 8.0 * L - 64.0
    direct = oracle.expcast_codes(Z, 0.0).astype(int)
    cast = oracle.exp_cast_codes(Z, 0.0).astype(int)
    assert abs(float(np.mean(direct == cast)) - g["value"]) < 0.003
    assert int(np.max(np.abs(direct - cast))) == g["max_code_distance"]


def test_baseline_rows_within_rounding_bound():
    q, k, v = _inputs(1, 700, 2, 41, bias=1.0, vdist="t3")
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rows_s = np.arange(0, 700, 19)
    rows_bh = np.arange(rows_s.size) % 2
    r = oracle.attention_rows(prep, rows_bh, rows_s, cast=True, mid_window=False)
    e = oracle.attention_rows(prep, rows_bh, rows_s)
    delta = 2.0 ** -4
    err_cast, err_expcast = [], []
    for i, (bh, s) in enumerate(zip(rows_bh, rows_s)):
        o_ref, z, vv = _exact_on_quantised(prep, bh, s)
        Z = 8.0 * z
        p = np.exp2((Z - Z.max()) / 8.0)
        tail = p[(Z - r["m8"][i]) / 8.0 + 8.0 < -6.0].sum() / p.sum()
        bound = (2.0 * delta / (1.0 - delta) + 2.0 * tail) * np.abs(vv).max()
        assert np.abs(r["out"][i] - o_ref).max() <= bound
        err_cast.append(np.linalg.norm(r["out"][i] - o_ref) / np.linalg.norm(o_ref))
        err_expcast.append(np.linalg.norm(e["out"][i] - o_ref) / np.linalg.norm(o_ref))
    # the two byte paths have errors of the same size (they agree within a code)
    ratio = float(np.mean(err_cast) / np.mean(err_expcast))
    assert 0.5 < ratio < 1.5, ratio
    assert not np.allclose(r["out"], e["out"])        # the flag is honoured


def test_baseline_block_codes_within_one_code_of_expcast():
    q, k, v = _inputs(1, 500, 1, 42)
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rng = np.random.default_rng(43)
    eq, n = 0, 0
    for s in rng.integers(0, 500, 12):
        m8 = float(rng.integers(-40, 40)) + (oracle.C0 + oracle.BETA) % 1.0
        for j in range(prep.nb):
            a = oracle.block_codes(prep, 0, int(s), j, m8).astype(int)
            b = oracle.block_codes(prep, 0, int(s), j, m8, cast=True).astype(int)
            assert np.abs(a - b).max() <= 1
            eq += int((a == b).sum())
            n += a.size
    assert eq / n > 0.7


def test_natural_order_visits_block_zero_first():
    q, k, v = _inputs(1, 1100, 1, 44)
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rows = np.arange(0, 1100, 61)
    r = oracle.attention_rows(prep, np.zeros_like(rows), rows, dump_block=0, mid_window=False, cast=True)
    tab = oracle.e4m3_table()
    frac = (oracle.C0 + oracle.BETA) % 1.0
    for i, s in enumerate(rows):
        kc = prep.kc[0, 0, :128]
        z = (tab[kc] @ tab[prep.qc[0, 0, s]]) * prep.sq[0, 0, s // 128] * prep.sk[0, 0, 0] * SM * math.log2(math.e)
        assert r["dump_m8"][i] == pytest.approx(math.ceil(8.0 * z.max() - frac) + frac, abs=1e-9)
        assert np.array_equal(r["codes"][i], oracle.block_codes(prep, 0, s, 0, r["dump_m8"][i], cast=True))

