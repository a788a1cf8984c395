"""Pins of the oracle's split key ranges (the short-sequence schedule: each
range of key blocks runs its own online softmax, then the partial results are
merged with the usual rescale-by-reference formula).

* With exact exp2 and no quantisation, any split count reproduces
  brute-force softmax attention in double: a dropped, repeated or mis-weighted
  range would break this.
* One range is the unsplit computation, bit for bit.
* With ExpCast, split rows stay within the 3.64% total-variation bound of
  exact attention on the same quantised inputs (VC-Attention summary,
  "ExpCast-FP8"), like unsplit rows.
"""
import numpy as np
import pytest

import oracle
from test_oracle_attention import GOLDEN, _bits, _exact_on_quantised, _inputs, _softmax_attention


@pytest.mark.parametrize("S", [129, 300, 513, 1000])
@pytest.mark.parametrize("nsplit", [2, 3, 5])
@pytest.mark.parametrize("mid", [1, 0])
def test_exact_split_equals_softmax_attention(S, nsplit, mid):
    nb = (S + 127) // 128
    if nsplit > nb:
        pytest.skip("more ranges than key blocks")
    rng = np.random.default_rng(S + 10 * nsplit)
    q = rng.standard_normal((1, S, 128)) * 2
    k = rng.standard_normal((1, S, 128)) * 2
    v = rng.standard_normal((1, S, 128))
    rows = np.arange(S)
    out, nres = oracle.attention_exact_rows(q, k, v, np.zeros_like(rows), rows, mid_window=mid, nsplit=nsplit)
    np.testing.assert_allclose(out, _softmax_attention(q[0], k[0], v[0]), rtol=1e-10, atol=1e-12)
    assert nres.min() >= nsplit          # every range sets its own reference at least once


def test_one_range_is_the_unsplit_computation():
    q, k, v = _inputs(1, 700, 2, 51, bias=1.0)
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rows = np.arange(0, 700, 13)
    bh = rows % 2
    a = oracle.attention_rows(prep, bh, rows)
    b = oracle.attention_rows(prep, bh, rows, nsplit=1)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["m8"], b["m8"])


@pytest.mark.parametrize("nsplit", [2, 4])
def test_expcast_split_rows_within_total_variation_bound(nsplit):
    q, k, v = _inputs(1, 700, 2, 52, bias=1.0, vdist="t3")
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rows_s = np.arange(0, 700, 17)
    rows_bh = np.arange(rows_s.size) % 2
    r = oracle.attention_rows(prep, rows_bh, rows_s, nsplit=nsplit)
    tv = GOLDEN["tv_bound"]["value"]
    for i, (bh, s) in enumerate(zip(rows_bh, rows_s)):
        o_ref, z, vv = _exact_on_quantised(prep, bh, s)
        Z = 8.0 * z
        p = np.exp2((Z - Z.max()) / 8.0)
        # underflow tail: mass below the normal range of the final reference
        # (a range with a lower reference of its own has less, not more)
        tail = p[(Z - r["m8"][i]) / 8.0 + 8.0 < -6.0].sum() / p.sum()
        assert np.abs(r["out"][i] - o_ref).max() <= 2.0 * (tv + tail) * np.abs(vv).max()


def test_split_arguments_are_checked():
    q, k, v = _inputs(1, 300, 1, 53)
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    rows = np.arange(3)
    with pytest.raises(ValueError):
        oracle.attention_rows(prep, np.zeros_like(rows), rows, nsplit=4)          # 3 key blocks
    with pytest.raises(ValueError):
        oracle.attention_rows(prep, np.zeros_like(rows), rows, nsplit=2, repair=oracle.Repair(prep, 0.1))
