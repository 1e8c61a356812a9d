"""Pins of the oracle's probabilistic drafting (Hybrid Spark sec. 4.5, App. H):
y ~ softmax(z / T) per draft row by inverse CDF in vocabulary order.

Closed forms on hand-built rows (the CDF steps of [1, 2, 3] / 6, and the
same rows at T = 1/2, where the odds square); a chi-square test of the drawn
frequencies over many steps; the counter domain of the uniforms, apart from
verification's; a row holding NaN drafts its argmax and is flagged."""
import math

import numpy as np
import pytest


def _row(weights):
    return np.log(np.asarray(weights, np.float64)).astype(np.float32).reshape(1, 1, -1)


@pytest.mark.parametrize("u,tok", [(0.0, 0), (0.1, 0), (0.17, 1), (0.49, 1), (0.51, 2), (0.99, 2)])
def test_inverse_cdf_steps(orc, u, tok):
    o = orc.sample_drafts(_row([1, 2, 3]), 1.0, u_override=[[u]])
    assert o.y[0, 0] == tok


@pytest.mark.parametrize("u,tok", [(0.07, 0), (0.08, 1), (0.35, 1), (0.36, 2)])
def test_temperature_half_squares_the_odds(orc, u, tok):
    # q = [1, 4, 9] / 14: steps at 1/14 = 0.0714 and 5/14 = 0.357
    o = orc.sample_drafts(_row([1, 2, 3]), 0.5, u_override=[[u]])
    assert o.y[0, 0] == tok
    np.testing.assert_allclose(o.q[0, 0], [1, 4, 9][tok] / 14, rtol=1e-6)


def test_draws_follow_q_chi_square(orc):
    rng = np.random.default_rng(3)
    z = (rng.standard_normal((2, 3, 8)) * 1.5).astype(np.float32)
    T = 0.8
    N = 4000
    counts = np.zeros((2, 3, 8))
    for step in range(N):
        o = orc.sample_drafts(z, T, seed=11, step=step)
        for r in range(2):
            for k in range(3):
                counts[r, k, o.y[r, k]] += 1
    for r in range(2):
        for k in range(3):
            q = np.exp(z[r, k] / T - np.max(z[r, k] / T))
            q /= q.sum()
            chi2 = ((counts[r, k] - N * q) ** 2 / (N * q)).sum()
            assert chi2 < 30.0, (r, k, chi2)  # 7 degrees of freedom: P(chi2 > 30) ~ 1e-4


def test_uniform_counter_domain(orc):
    z = np.zeros((3, 4, 5), np.float32)
    o = orc.sample_drafts(z, 1.0, seed=(5 << 32) | 7, step=(2 << 32) | 9)
    for r in range(3):
        for k in range(1, 5):
            w = orc.philox4x32_10([r, 0x40000000 + k, 9, 2], [7, 5])
            assert o.u[r, k - 1] == (w[0] >> 8) / 2 ** 24
            assert o.u[r, k - 1] != orc.round_uniforms(((5 << 32) | 7), ((2 << 32) | 9), r, k)[0]


def test_nonfinite_row_drafts_its_argmax(orc):
    z = np.array([[[0.0, 3.0, np.nan, 1.0], [0.0, 0.0, 0.0, 0.0]]], np.float32)
    o = orc.sample_drafts(z, 1.0, seed=1)
    assert o.status & orc.ST_NONFINITE and o.y[0, 0] == 1
