"""Pins of the oracle's FP32-defined quantisation and of the repair selection.

The quantised codes are checked against torch's float8_e4m3fn cast of the
FP32 product x * (448 / amax), the scales against numpy's amax, the residual
energy against its defining sum in double, and the top-n selection against a
brute-force sort.  ("Open VC Attention" catalogue entry: per-block Q/K scales,
per-head V scale; prepare_v_repair(budget).)
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _cast(x32):
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _f32(t):
    return t.to(torch.float32).numpy()


@pytest.mark.parametrize("S", [1, 127, 128, 129, 300])
def test_quantize_blocks_scales_codes_and_tail(S):
    rng = np.random.default_rng(S)
    B, H = 2, 3
    x = _bf16(rng.standard_normal((B, S, H, 128)) * 3 + rng.standard_normal((1, 1, H, 128)))
    codes, scales = oracle.quantize_blocks(_bits(x))
    nb = (S + 127) // 128
    xf = _f32(x)
    for b in range(B):
        for h in range(H):
            for j in range(nb):
                blk = xf[b, j * 128:(j + 1) * 128, h, :]
                amax = np.float32(np.abs(blk).max())
                assert scales[b, h, j] == np.float32(amax / np.float32(448.0))
                r = np.float32(448.0) / amax
                want = _cast(blk * r)
                got = codes[b, h, j * 128:j * 128 + blk.shape[0]]
                assert np.array_equal(got, want)
                assert not codes[b, h, j * 128 + blk.shape[0]:(j + 1) * 128].any()


def test_quantize_blocks_zero_block_has_unit_scale():
    x = torch.zeros((1, 256, 1, 128), dtype=torch.bfloat16)
    x[0, 130, 0, 5] = 2.0
    codes, scales = oracle.quantize_blocks(_bits(x))
    assert scales[0, 0, 0] == 1.0 and not codes[0, 0, :128].any()
    assert scales[0, 0, 1] == np.float32(2.0 / 448.0)
    assert codes[0, 0, 130, 5] == 0x7E


def test_quantize_v_per_head_scale_and_layout():
    rng = np.random.default_rng(7)
    B, S, H = 1, 200, 2
    v = _bf16(rng.standard_t(3, (B, S, H, 128)))
    codes, sv, energy = oracle.quantize_v(_bits(v))
    vf = _f32(v)
    for h in range(H):
        amax = np.float32(np.abs(vf[0, :, h]).max())
        assert sv[0, h] == np.float32(amax / np.float32(448.0))
        assert np.array_equal(codes[0, h, :S], _cast(vf[0, :, h] * (np.float32(448.0) / amax)))
        assert not codes[0, h, S:].any()


def test_residual_energy_is_the_squared_residual_norm():
    rng = np.random.default_rng(8)
    B, S, H = 1, 64, 2
    v = _bf16(rng.standard_normal((B, S, H, 128)))
    codes, sv, energy = oracle.quantize_v(_bits(v))
    vf = _f32(v).astype(np.float64)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for h in range(H):
        R = vf[0, :, h] - np.float64(sv[0, h]) * dec[0, h, :S]
        e_ref = (R * R).sum(axis=1)
        np.testing.assert_allclose(energy[0, h], e_ref, rtol=2e-5, atol=1e-30)


def test_residual_energy_zero_for_representable_values():
    # amax = 448 -> s_v = 1, and every value is an E4M3 (and BF16) value.
    tab = oracle.e4m3_table()
    vals = tab[np.r_[1:127, 129:255]]
    rng = np.random.default_rng(9)
    v = rng.choice(vals, (1, 40, 1, 128)).astype(np.float32)
    v[0, 0, 0, 0] = 448.0
    codes, sv, energy = oracle.quantize_v(_bits(_bf16(v)))
    assert sv[0, 0] == 1.0
    assert not energy.any()


def test_residual_energy_order_and_nonnegativity():
    rng = np.random.default_rng(10)
    R = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3, 128)).astype(np.float32)
    e = oracle.residual_energy(R)
    assert e >= 0
    assert e == pytest.approx(float((R.astype(np.float64) ** 2).sum()), rel=1e-5)
    assert oracle.residual_energy(np.zeros(128, np.float32)) == 0.0


@pytest.mark.parametrize("S,budget,n", [(73397, 0.005, 367), (73397, 0.01, 734),
                                        (73397, 0.02, 1468), (1000, 0.0001, 1), (10, 1.0, 10)])
def test_repair_count_is_ceil_budget_times_s(S, budget, n):
    assert oracle.repair_count(S, budget) == n


def test_repair_select_matches_brute_force_with_ties():
    rng = np.random.default_rng(11)
    B, H, S = 2, 3, 500
    e = rng.integers(0, 40, (B, H, S)).astype(np.float32)      # many ties
    for n in (1, 7, 64, 500):
        idx = oracle.repair_select(e, n)
        for b in range(B):
            for h in range(H):
                order = np.lexsort((np.arange(S), -e[b, h].astype(np.float64)))
                assert np.array_equal(idx[b, h], np.sort(order[:n]))


def test_repair_quantize_scale_and_codes():
    rng = np.random.default_rng(12)
    B, S, H = 1, 300, 2
    v = _bf16(rng.standard_normal((B, S, H, 128)))
    vc, sv, energy = oracle.quantize_v(_bits(v))
    n = oracle.repair_count(S, 0.05)
    idx = oracle.repair_select(energy, n)
    dcodes, sr = oracle.repair_quantize(_bits(v), vc, sv, idx)
    vf = _f32(v)
    dec = torch.from_numpy(vc).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for h in range(H):
        t = idx[0, h]
        R = vf[0, t, h] - (sv[0, h] * dec[0, h, t]).astype(np.float32)
        amax = np.float32(np.abs(R).max())
        assert sr[0, h] == np.float32(amax / np.float32(448.0))
        assert np.array_equal(dcodes[0, h], _cast(R * (np.float32(448.0) / amax)))
        # the selected tokens carry the largest energies
        assert energy[0, h, t].min() >= np.delete(energy[0, h], t).max()


def test_half_decoder_matches_ieee_binary16_on_every_pattern():
    """The oracle's FP16 decoder (written from the format definition) against
    numpy's binary16 on all 65536 bit patterns; NaNs as NaNs."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_bits_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_fp16_and_bf16_inputs_quantise_alike_on_shared_values():
    """Values exact in both formats give the same codes, scales and energies
    through the FP16 and the BF16 paths ("Open VC Attention" catalogue entry:
    FP16 or BF16 inputs)."""
    rng = np.random.default_rng(11)
    # m * 2^e with |m| < 128, -6 <= e <= 2: at most 8 significant bits (exact
    # in BF16) and inside FP16's normal range
    m = rng.integers(-127, 128, (1, 200, 2, 128)).astype(np.float64)
    e = rng.integers(-6, 3, (1, 200, 2, 128))
    x = np.ldexp(m, e).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xh = torch.from_numpy(x).to(torch.float16)
    assert np.array_equal(xb.float().numpy(), x) and np.array_equal(xh.float().numpy(), x)
    cb, sb = oracle.quantize_blocks(_bits(xb))
    ch, sh = oracle.quantize_blocks(_bits(xh), fp16=True)
    assert np.array_equal(cb, ch) and np.array_equal(sb, sh)
    vb = oracle.quantize_v(_bits(xb))
    vh = oracle.quantize_v(_bits(xh), fp16=True)
    for a, b in zip(vb, vh):
        assert np.array_equal(a, b)
    # and they differ once the bits are misread: the flag is honoured
    cx, _ = oracle.quantize_blocks(_bits(xh))
    assert not np.array_equal(cx, ch)


def test_k_mean_is_the_channel_mean_to_fp32_rounding():
    """K smoothing's channel means against float64 means (sum of S terms in
    FP32: error below S * 2^-23 * max|partial|), and exact on tiny inputs."""
    rng = np.random.default_rng(5)
    for S in (1, 2, 3, 129, 1000):
        x = _bf16(rng.standard_normal((2, S, 3, 128)) + 4.0 * rng.standard_normal((1, 1, 3, 128)))
        mean = oracle.k_mean(_bits(x))
        xf = _f32(x).astype(np.float64)
        ref = xf.mean(axis=1)                           # [B, H, 128]
        bound = S * 2.0 ** -23 * (np.abs(xf).sum(axis=1) / S + 1e-30) * 2
        assert np.all(np.abs(mean - ref) <= bound + 1e-12)
        if S <= 2:       # a sum of at most 2 BF16 values is exact in FP32, and so is /1 or /2
            assert np.array_equal(mean, ref.astype(np.float32))


def test_smoothed_k_codes_are_casts_of_the_centred_values():
    """quantize_blocks(x, mean): codes equal torch's E4M3 casts of
    fl(fl(x - mean) * 448/amax) with amax over the centred block."""
    rng = np.random.default_rng(8)
    S, H = 300, 2
    x = _bf16(rng.standard_normal((1, S, H, 128)) + 5.0 * rng.standard_normal((1, 1, H, 128)))
    mean = oracle.k_mean(_bits(x))
    codes, scales = oracle.quantize_blocks(_bits(x), mean=mean)
    xc = (_f32(x) - mean[:, None, :, :]).astype(np.float32)
    for h in range(H):
        for j in range(3):
            blk = xc[0, j * 128:(j + 1) * 128, h, :]
            amax = np.float32(np.abs(blk).max())
            assert scales[0, h, j] == np.float32(amax / np.float32(448.0))
            assert np.array_equal(codes[0, h, j * 128:j * 128 + blk.shape[0]], _cast(blk * (np.float32(448.0) / amax)))
    # the offset no longer sets the scale: centred blocks use finer steps
    _, raw_scales = oracle.quantize_blocks(_bits(x))
    assert np.all(scales < raw_scales)
