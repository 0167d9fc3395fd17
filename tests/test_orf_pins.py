"""Pins for the oracle's orthogonal-random-feature draw (CPU only).

The FAVOR+ projection of "Sub-Linear Memory: How to Make Performers SLiM",
section 2.1, is redrawn on the device from a counter-based generator; the
oracle (oracle/orf.py) restates the same published generator and recipe.
Here it is pinned against what fixes it from outside: the generator's
published known-answer vectors, the moments of the Gaussians it makes, the
orthogonality of each block and the chi_d law of the feature lengths.
"""
import json
import os

import numpy as np
import pytest

from oracle import orf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answer_vectors():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    for vec in kat["vectors"]:
        ctr = np.array([int(x, 16) for x in vec["counter"]], dtype=np.uint64)
        key = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint64)
        out = orf.philox4x32_10(ctr, key)
        assert ["%08x" % int(x) for x in out] == vec["out"]


def test_gaussians_have_unit_normal_moments():
    g = np.concatenate([orf.block_gaussians(7, 0, i, b, 1 << 14) for i in range(4) for b in range(4)])
    n = g.size
    assert abs(g.mean()) < 4 / np.sqrt(n)
    assert abs(g.var() - 1.0) < 4 * np.sqrt(2.0 / n)
    assert abs(np.mean(g ** 4) - 3.0) < 4 * np.sqrt(96.0 / n)  # kurtosis of N(0, 1)
    # Kolmogorov-Smirnov distance to the normal CDF, far inside its 0.1% band
    from math import erf, sqrt
    xs = np.sort(g[:20000])
    cdf = np.array([0.5 * (1 + erf(x / sqrt(2))) for x in xs])
    emp = np.arange(1, xs.size + 1) / xs.size
    assert np.max(np.abs(cdf - emp)) < 1.95 / np.sqrt(xs.size)


@pytest.mark.parametrize("d,m", [(16, 32), (64, 256), (64, 100), (128, 128)])
def test_blocks_are_orthogonal_with_chi_lengths(d, m):
    w = orf.orf_matrix(d, m, seed=1234, step=3, i=1)
    assert w.shape == (d, m)
    lengths = np.linalg.norm(w, axis=0)
    for b0 in range(0, m, d):
        blk = w[:, b0:b0 + d]
        gram = blk.T @ blk
        np.testing.assert_allclose(gram, np.diag(np.diag(gram)), atol=1e-10 * np.max(gram))
    # the lengths themselves: the norms of the block's second d*d Gaussians
    g = orf.block_gaussians(1234, 3, 1, 0, 2 * d * d)
    np.testing.assert_allclose(lengths[:min(d, m)], np.linalg.norm(g[d * d:].reshape(d, d), axis=0)[:min(d, m)],
                               rtol=1e-12)


def test_lengths_follow_chi_d():
    d = 32
    w = orf.orf_matrices(16, d, 128, seed=99)
    sq = np.sum(w ** 2, axis=1).ravel()  # squared lengths: chi-square with d degrees
    n = sq.size
    assert abs(sq.mean() - d) < 4 * np.sqrt(2.0 * d / n)
    assert abs(sq.var() - 2 * d) < 4 * np.sqrt((48.0 * d + 12.0 * d * d) / n)


def test_directions_are_the_positive_diagonal_qr():
    """Block 0's directions are G's unique QR factor with diag(R) > 0: Q^T G
    is upper triangular with a positive diagonal."""
    d = 16
    w = orf.orf_matrix(d, d, seed=5)
    q = w / np.linalg.norm(w, axis=0)[None, :]
    g = orf.block_gaussians(5, 0, 0, 0, 2 * d * d)[:d * d].reshape(d, d)
    r = q.T @ g
    assert np.max(np.abs(np.tril(r, -1))) < 1e-12 * np.max(np.abs(r))
    assert np.all(np.diag(r) > 0)


def test_redraws_are_deterministic_and_distinct():
    a = orf.orf_matrices(3, 16, 48, seed=42, step=0)
    np.testing.assert_array_equal(a, orf.orf_matrices(3, 16, 48, seed=42, step=0))
    b = orf.orf_matrices(3, 16, 48, seed=42, step=1)
    assert np.max(np.abs(a - b)) > 0.1
    assert np.max(np.abs(a[0] - a[1])) > 0.1  # matrices of one redraw differ


def test_per_head_w_is_each_head_with_its_own_w():
    """W per head: head h is exactly the shared-W computation with W = w[h];
    equal matrices give the shared-W result and dW sums per head."""
    import oracle

    rng = np.random.default_rng(61)
    b, h, length, d, m = 2, 3, 20, 4, 8
    q, k, v, dy = (rng.standard_normal((b, h, length, d)) * 0.6 for _ in range(4))
    w = orf.orf_matrices(h, d, m, seed=3)
    y = oracle.recurrence_forward(q, k, v, w)
    dq, dk, dv, dw = oracle.recurrence_backward(q, k, v, w, dy)
    assert dw.shape == (h, d, m)
    for hh in range(h):
        sl = lambda t: t[:, hh:hh + 1]
        np.testing.assert_array_equal(y[:, hh:hh + 1], oracle.recurrence_forward(sl(q), sl(k), sl(v), w[hh]))
        ref = oracle.recurrence_backward(sl(q), sl(k), sl(v), w[hh], sl(dy))
        for got, exp in zip((dq, dk, dv), ref[:3]):
            np.testing.assert_array_equal(got[:, hh:hh + 1], exp)
        np.testing.assert_allclose(dw[hh], ref[3], rtol=1e-12)
    same = np.stack([w[0]] * h)
    np.testing.assert_allclose(oracle.recurrence_backward(q, k, v, same, dy)[3].sum(axis=0),
                               oracle.recurrence_backward(q, k, v, w[0], dy)[3], rtol=1e-11)
