"""Pins of the oracle's V-Smooth (VC-Attention summary, "V-Smooth": each
128-token block subtracts its mean, only the residual is quantised, and the
mean is added back through the row sums that online softmax keeps).

* The block mean is the mean: the residuals of a block sum to ~0 (up to the
  BF16 rounding of the mean).
* Reconstruction: s dec(code) + mu_b equals v within the E4M3 rounding of
  the residual plus the BF16 rounding of the mean.
* With values whose blocks are constant powers of two, both V-Smooth and the
  plain per-head V quantisation reproduce V exactly, so the two attention
  outputs must agree to rounding: the restore term enters with the right
  block and the right row-sum weight.
* On values with large per-block offsets (the case the method targets) V's
  reconstruction error drops by an order of magnitude and the attention
  error by its V part; on zero-mean values it stays about the same.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_attention import _bits, _inputs, _softmax_attention

SM = 1.0 / math.sqrt(128.0)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _blocks(S):
    return [(j * 128, min(S, j * 128 + 128)) for j in range((S + 127) // 128)]


@pytest.mark.parametrize("S", [1, 127, 300])
def test_residuals_of_a_block_sum_to_zero(S):
    rng = np.random.default_rng(S)
    v = rng.standard_normal((1, S, 2, 128)) * 3 + rng.standard_normal((1, 1, 2, 128)) * 5
    vb = _bf16(v)
    codes, sv, mu = oracle.vsmooth_v(_bits(vb))
    x = vb.float().numpy()
    for h in range(2):
        for j, (t0, t1) in enumerate(_blocks(S)):
            R = x[0, t0:t1, h, :] - mu[0, h, j]
            # |sum R| <= n * (half a BF16 ulp of the mean) + FP32 rounding
            ulp = np.spacing(np.abs(mu[0, h, j]).astype(np.float32)) * 2 ** 16
            bound = (t1 - t0) * (ulp / 2 + 1e-5 * np.abs(x[0, t0:t1, h, :]).max(axis=0)) + 1e-6
            assert np.all(np.abs(R.sum(axis=0)) <= bound)


def test_reconstruction_within_rounding_bounds():
    rng = np.random.default_rng(5)
    S = 700
    v = rng.standard_t(3, (1, S, 2, 128)) + 4.0 * rng.standard_normal((1, S // 128 + 1, 2, 128)).repeat(128, 1)[:, :S]
    vb = _bf16(v)
    codes, sv, mu = oracle.vsmooth_v(_bits(vb))
    tab = oracle.e4m3_table()
    x = vb.float().numpy()
    for h in range(2):
        s = float(sv[0, h])
        mub = np.repeat(mu[0, h], 128, axis=0)[:S].astype(np.float64)
        rec = s * tab[codes[0, h, :S]] + mub
        R = np.abs(x[0, :, h, :] - mub)
        # E4M3 keeps 3 mantissa bits: half an ulp is <= 2^-4 of |R| (normal
        # range) or 2^-10 s (subnormal); the residual is taken against the
        # stored mean, so the mean adds no error of its own
        bound = 2.0 ** -4 * R + 2.0 ** -10 * s + 1e-6
        assert np.all(np.abs(rec - x[0, :, h, :]) <= bound)
    # the residual's amax sets the scale: some code is the largest, 126 (448)
    assert (codes & 0x7F).max() == 126


def test_exact_values_give_the_plain_result():
    """Blocks of constant values +-7 * 2^k with amax 28: the plain per-head
    scale s = 28/448 = 2^-4 and r = 16 are exact and every value is an E4M3
    code times s, and V-Smooth's residual is exactly 0 (s = 1, mu_b = the
    block's value), so both paths reconstruct V exactly."""
    rng = np.random.default_rng(7)
    S = 600
    nb = (S + 127) // 128
    q, k, _ = _inputs(1, S, 1, 71)
    c = np.ldexp(7.0 * rng.choice([-1.0, 1.0], (nb, 128)), rng.integers(-4, 3, (nb, 128)))
    c[0, 0] = 28.0
    v = np.repeat(c, 128, axis=0)[:S][None, :, None, :]
    vb = _bf16(v)
    plain = oracle.Prepared(_bits(q), _bits(k), _bits(vb))
    smooth = oracle.Prepared(_bits(q), _bits(k), _bits(vb), v_smooth=True)
    assert not smooth.vc.any() and np.all(smooth.sv == 1.0)        # residual exactly 0
    assert plain.sv[0, 0] == 2.0 ** -4
    rows = np.arange(0, S, 7)
    a = oracle.attention_rows(plain, np.zeros_like(rows), rows)
    b = oracle.attention_rows(smooth, np.zeros_like(rows), rows)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(a["m8"], b["m8"])


def _err(prep, q, k, v, rows):
    out = oracle.attention_rows(prep, np.zeros_like(rows), rows)["out"]
    qq, kk, vv = (x.float().numpy()[0, :, 0, :].astype(np.float64) for x in (q, k, v))
    ref = _softmax_attention(qq[rows], kk, vv)
    return float(np.linalg.norm(out - ref) / np.linalg.norm(ref))


def test_v_smooth_cuts_the_error_of_block_offsets():
    rng = np.random.default_rng(8)
    S = 1000
    q, k, _ = _inputs(1, S, 1, 81)
    offs = 20.0 * rng.standard_normal(((S + 127) // 128, 128))
    v = (np.repeat(offs, 128, axis=0)[:S] + rng.standard_normal((S, 128)))[None, :, None, :]
    vb = _bf16(v)
    rows = np.arange(0, S, 9)
    plain = oracle.Prepared(_bits(q), _bits(k), _bits(vb))
    smooth = oracle.Prepared(_bits(q), _bits(k), _bits(vb), v_smooth=True)
    # V itself: the reconstruction error drops by an order of magnitude
    tab = oracle.e4m3_table()
    x = vb.float().numpy()[0, :, 0, :]
    rec_plain = plain.sv[0, 0] * tab[plain.vc[0, 0, :S]]
    rec_smooth = smooth.sv[0, 0] * tab[smooth.vc[0, 0, :S]] + np.repeat(smooth.vmu[0, 0], 128, axis=0)[:S]
    ev_plain = np.linalg.norm(rec_plain - x) / np.linalg.norm(x)
    ev_smooth = np.linalg.norm(rec_smooth - x) / np.linalg.norm(x)
    assert ev_smooth < 0.1 * ev_plain, (ev_smooth, ev_plain)
    # the attention output: the V part of the error goes, the P and QK parts stay
    e_plain = _err(plain, q, k, vb, rows)
    e_smooth = _err(smooth, q, k, vb, rows)
    assert e_smooth < 0.85 * e_plain, (e_smooth, e_plain)


def test_v_smooth_on_zero_mean_values_is_about_the_same():
    q, k, v = _inputs(1, 1000, 1, 82)
    rows = np.arange(0, 1000, 9)
    e_plain = _err(oracle.Prepared(_bits(q), _bits(k), _bits(v)), q, k, v, rows)
    e_smooth = _err(oracle.Prepared(_bits(q), _bits(k), _bits(v), v_smooth=True), q, k, v, rows)
    assert 0.7 * e_plain < e_smooth < 1.3 * e_plain


def test_v_smooth_excludes_repair():
    q, k, v = _inputs(1, 300, 1, 83)
    plain = oracle.Prepared(_bits(q), _bits(k), _bits(v))
    smooth = oracle.Prepared(_bits(q), _bits(k), _bits(v), v_smooth=True)
    rows = np.arange(3)
    with pytest.raises(ValueError):
        oracle.attention_rows(smooth, np.zeros_like(rows), rows, repair=oracle.Repair(plain, 0.1))
