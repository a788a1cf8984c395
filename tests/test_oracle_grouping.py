"""Pins of the oracle's V-Smooth grouping (VC-Attention summary, "V-Smooth":
online k-means clusters each head's value tokens, and keys and values are
permuted together, which leaves non-causal attention unchanged).

Checked against what Lloyd's algorithm fixes, recomputed here in float64:
* the permutation is a permutation, ordered by (cluster, index);
* every token's cluster is a nearest centroid among those the last
  assignment used;
* each update is the mean of the cluster's tokens (empty clusters keep their
  centroid);
* the k-means objective does not increase from one iteration to the next;
* on values drawn around a few centres in random order, grouping lets the
  block means of V-Smooth take out more of V, so V's reconstruction error
  drops clearly below V-Smooth without grouping.
"""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_attention import _bits, _inputs


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _clustered_v(S, H, centres, seed, noise=0.3):
    rng = np.random.default_rng(seed)
    c = rng.standard_normal((H, centres, 128)) * 4.0
    lab = rng.integers(0, centres, (S, H))
    v = c[np.arange(H)[None, :], lab] + noise * rng.standard_normal((S, H, 128))
    return _bf16(v[None]), lab


def _x(vb, h):
    return vb.float().numpy()[0, :, h, :].astype(np.float64)


@pytest.mark.parametrize("S,C", [(1, 1), (200, 7), (700, 16)])
def test_permutation_is_ordered_by_cluster_then_index(S, C):
    vb, _ = _clustered_v(S, 2, 5, S)
    labels, cent, perm = oracle.kmeans_group(_bits(vb), C, 3)
    for h in range(2):
        p = perm[0, h]
        assert np.array_equal(np.sort(p), np.arange(S))
        key = labels[0, h][p].astype(np.int64) * S + p
        assert np.all(np.diff(key) > 0)


def test_first_centroids_are_the_spread_tokens():
    """Before any update (one assignment step) the centroids are the tokens
    floor(c S / C)."""
    vb, _ = _clustered_v(500, 2, 4, 10)
    _, cent, _ = oracle.kmeans_group(_bits(vb), 9, 1)
    for h in range(2):
        assert np.array_equal(cent[0, h], _x(vb, h)[(np.arange(9) * 500) // 9])


def test_assignment_is_a_nearest_centroid():
    vb, _ = _clustered_v(900, 2, 6, 11)
    labels, cent, _ = oracle.kmeans_group(_bits(vb), 12, 3)
    for h in range(2):
        x, mu = _x(vb, h), cent[0, h].astype(np.float64)
        d = ((x[:, None, :] - mu[None, :, :]) ** 2).sum(-1)
        chosen = d[np.arange(len(x)), labels[0, h]]
        # the oracle's distances are the same double sums: exactly the minimum,
        # and ties go to the lower cluster
        assert np.all(chosen <= d.min(axis=1) * (1 + 1e-12))
        first = np.argmax(d <= d.min(axis=1, keepdims=True) * (1 + 1e-12), axis=1)
        assert np.array_equal(labels[0, h], first)


def test_update_is_the_mean_and_the_objective_never_rises():
    vb, _ = _clustered_v(1000, 1, 5, 12, noise=1.0)
    x = _x(vb, 0)
    J = []
    prev = None
    for it in range(1, 7):
        labels, cent, _ = oracle.kmeans_group(_bits(vb), 8, it)
        lab, mu = labels[0, 0], cent[0, 0].astype(np.float64)
        J.append(((x - mu[lab]) ** 2).sum())
        if prev is not None:
            plab, pmu = prev
            for c in range(8):
                m = plab == c
                want = x[m].mean(axis=0) if m.any() else pmu[c]
                np.testing.assert_allclose(mu[c], want, rtol=1e-12, atol=1e-12)
        prev = (lab, mu)
    assert all(b <= a * (1 + 1e-12) for a, b in zip(J, J[1:])), J
    assert J[-1] < J[0]


def test_grouping_lets_block_means_take_out_clustered_values():
    S, H = 2048, 1
    vb, _ = _clustered_v(S, H, 12, 13, noise=0.2)
    tab = oracle.e4m3_table()
    x = vb.float().numpy()[0, :, 0, :]

    def v_error(v_bits):
        codes, sv, mu = oracle.vsmooth_v(v_bits)
        return sv[0, 0] * tab[codes[0, 0, :S]] + np.repeat(mu[0, 0], 128, axis=0)[:S]

    plain_err = np.linalg.norm(v_error(_bits(vb)) - x) / np.linalg.norm(x)
    _, _, perm = oracle.kmeans_group(_bits(vb), 16, 4)
    vp = oracle.permute_tokens(_bits(vb), perm)
    xg = x[perm[0, 0]]
    grouped_err = np.linalg.norm(v_error(vp) - xg) / np.linalg.norm(xg)
    # clusters of ~170 tokens straddle block boundaries and the residual scale
    # is one per head, so not all of V goes; at least a quarter of the error does
    assert grouped_err < 0.75 * plain_err, (grouped_err, plain_err)


def test_grouped_prepared_tensors_are_the_permuted_ones():
    q, k, v = _inputs(1, 300, 2, 14)
    _, _, perm = oracle.kmeans_group(_bits(v), 4, 2)
    a = oracle.Prepared(_bits(q), _bits(k), _bits(v), v_smooth=True, perm=perm)
    kp, vp = oracle.permute_tokens(_bits(k), perm), oracle.permute_tokens(_bits(v), perm)
    b = oracle.Prepared(_bits(q), kp, vp, v_smooth=True)
    assert np.array_equal(a.kc, b.kc) and np.array_equal(a.vc, b.vc) and np.array_equal(a.qc, b.qc)
    with pytest.raises(ValueError):
        oracle.kmeans_group(_bits(v), 301, 2)
