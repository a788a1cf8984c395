"""Pins of the oracle's Q smoothing (VC-Attention summary, "Why attention is
the video bottleneck": the prior low-bit kernels smooth Q and K before
quantising them).

Subtracting Q's channel mean mu_q changes every score of a row by
mu_q . k_j, a term that differs from key to key, so unlike K smoothing it
must be added back: the oracle gives key t the bias beta_t = mu_q . dec(K^_t)
and each score gains s_k beta_t (times the softmax scale).

* Exact skeleton: with exact exponentials and no quantisation, q - mu plus
  the bias mu . k_t equals plain softmax attention of q to 1e-10, whatever mu
  is (so the bias has the right sign, factor and key).
* Quantised scores: the codes the oracle writes for a smoothed query row are
  the ExpCast codes of the exact product of the dequantised vectors,
  (mu_q + s_q dec(Q^'_i)) . (s_k dec(K^_j)), computed here independently.
* Zero-mean queries: mu_q = 0 exactly, and the smoothed path equals the
  plain one exactly.
* On queries with a per-channel offset (the workloads' bias N(0, var 2)),
  smoothing Q as well as K lowers the error against exact attention further.
"""
import math

import numpy as np
import torch

import oracle
from test_oracle_attention import SM, _bits, _inputs, _softmax_attention

LOG2E = 1.0 / math.log(2.0)


def test_bias_restores_exact_attention():
    rng = np.random.default_rng(31)
    BH, S = 2, 300
    q = rng.standard_normal((BH, S, 128)) + 3.0 * rng.standard_normal((BH, 1, 128))
    k = rng.standard_normal((BH, S, 128)) + 2.0 * rng.standard_normal((BH, 1, 128))
    v = rng.standard_normal((BH, S, 128))
    mu = q.mean(axis=1, keepdims=True) + 0.25 * rng.standard_normal((BH, 1, 128))   # any offset
    kbias = np.einsum("btd,bd->bt", k, mu[:, 0])
    bh, s = np.meshgrid(np.arange(BH), np.arange(S), indexing="ij")
    out, _ = oracle.attention_exact_rows(q - mu, k, v, bh.ravel(), s.ravel(), kbias=kbias)
    for b in range(BH):
        np.testing.assert_allclose(out[b * S:(b + 1) * S], _softmax_attention(q[b], k[b], v[b]),
                                   rtol=1e-10, atol=1e-12)
    # without the bias the result is a different attention
    out0, _ = oracle.attention_exact_rows(q - mu, k, v, bh.ravel(), s.ravel())
    assert np.abs(out0 - out).max() > 1e-2


def test_codes_are_those_of_the_exact_product_of_the_dequantised_vectors():
    q, k, v = _inputs(1, 700, 2, 32, bias=np.sqrt(2.0))
    prep = oracle.Prepared(_bits(q), _bits(k), _bits(v), smooth_q=True, smooth_k=True)
    tab = oracle.e4m3_table()
    mu = prep.qmean.astype(np.float64)
    n_equal = n_total = 0
    for bh, row, j, m8 in ((0, 5, 2, 40.65), (1, 300, 5, -12.35), (1, 699, 0, 3.65), (0, 128, 3, 100.65)):
        qb = row // 128
        qv = prep.sq[0, bh, qb] * tab[prep.qc[0, bh, row]] + mu[0, bh]
        t = np.arange(j * 128, min(700, j * 128 + 128))
        kv = prep.sk[0, bh, j] * tab[prep.kc[0, bh, t]]
        Z = 8.0 * LOG2E * SM * (kv @ qv)
        want = oracle.expcast_codes(Z, m8)
        got = oracle.block_codes(prep, bh, row, j, m8)
        n_equal += int(np.sum(got[:t.size] == want))
        n_total += t.size
        assert np.abs(got[:t.size].astype(int) - want.astype(int)).max() <= 1
        assert not got[t.size:].any()
    assert n_equal == n_total


def test_zero_mean_queries_give_the_plain_result():
    q, k, v = _inputs(1, 256, 2, 33)
    qh = q.float().numpy()
    qz = np.concatenate([qh[:, :128], -qh[:, :128]], axis=1)          # channel means exactly 0
    qz = torch.from_numpy(qz).to(torch.bfloat16)
    plain = oracle.Prepared(_bits(qz), _bits(k), _bits(v))
    smooth = oracle.Prepared(_bits(qz), _bits(k), _bits(v), smooth_q=True)
    assert not smooth.qmean.any() and not smooth.kbias.any()
    assert np.array_equal(plain.qc, smooth.qc)
    rows = np.arange(0, 256, 5)
    a = oracle.attention_rows(plain, rows % 2, rows)
    b = oracle.attention_rows(smooth, rows % 2, rows)
    assert np.array_equal(a["out"], b["out"])


def test_q_smoothing_reduces_error_on_biased_queries():
    q, k, v = _inputs(1, 1024, 2, 34, bias=np.sqrt(2.0))
    qf, kf, vf = (x.to(torch.float64).numpy() for x in (q, k, v))
    rows_s = np.arange(0, 1024, 11)
    rows_bh = np.arange(rows_s.size) % 2
    ref = np.stack([_softmax_attention(qf[0, :, bh], kf[0, :, bh], vf[0, :, bh])[s]
                    for bh, s in zip(rows_bh, rows_s)])
    errs = []
    for sk, sq in ((False, False), (True, False), (True, True)):
        prep = oracle.Prepared(_bits(q), _bits(k), _bits(v), smooth_k=sk, smooth_q=sq)
        out = oracle.attention_rows(prep, rows_bh, rows_s)["out"]
        errs.append(np.linalg.norm(out - ref) / np.linalg.norm(ref))
    assert errs[1] < errs[0] and errs[2] < 0.9 * errs[1], errs
