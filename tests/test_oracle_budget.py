"""Pins of the oracle's budget sizing (Hybrid Spark sec. 2 adaptive
verification, sec. 4.3 Eq. (2), sec. 4.4, App. F linear cost model).

b* maximises G(b) = (batch + sum of the b largest survivals) / (C0 + p b),
lambda = G(b*) p.  Checked against exact rational arithmetic on small inputs,
the closed form of equal survivals, Eq. (2)'s rule that a slot raises goodput
only when its survival exceeds lambda, monotonicity in the slot cost, and
which slots count."""
from fractions import Fraction

import numpy as np
import pytest


def _exact(S, chain_len, mvl, C0, p):
    B, L = S.shape
    s = sorted((Fraction(float(S[r, k])) for r in range(B) for k in range(min(chain_len[r], mvl, L))),
               reverse=True)
    C0, p = Fraction(C0), Fraction(p)
    A, best, bs = Fraction(B), Fraction(B) / C0, 0
    for b in range(1, len(s) + 1):
        A += s[b - 1]
        G = A / (C0 + p * b)
        if G > best:
            best, bs = G, b
    return bs, best * p


@pytest.mark.parametrize("seed", range(20))
def test_budget_against_exact_rationals(orc, seed):
    rng = np.random.default_rng(seed)
    B, L = int(rng.integers(1, 9)), 7
    S = np.sort(rng.random((B, L)).astype(np.float32), axis=1)[:, ::-1]  # survivals fall along a chain
    S = np.cumprod(S, axis=1).astype(np.float32)
    chain_len = rng.integers(0, L + 1, B).astype(np.int32)
    mvl = int(rng.integers(1, L + 1))
    C0, p = float(rng.uniform(1, 20)), float(rng.uniform(0.05, 2))
    o = orc.size_budget(S, chain_len, mvl, C0, p)
    b, lam = _exact(S, chain_len, mvl, C0, p)
    assert o.b_star == b
    assert abs(o.lam - float(lam)) <= 1e-12 * float(lam)


@pytest.mark.parametrize("s,C0,p", [(0.8, 10.0, 1.0), (0.05, 10.0, 1.0), (0.5, 4.0, 2.0), (0.5, 8.0, 1.0)])
def test_equal_survivals_closed_form(orc, s, C0, p):
    B, L = 4, 5
    S = np.full((B, L), s, np.float32)
    o = orc.size_budget(S, np.full(B, L, np.int32), L, C0, p)
    # G(b) = (B + b s) / (C0 + p b) is monotone in b: all slots if s/p > B/C0,
    # none otherwise (s/p = B/C0 makes G constant: the smallest b wins)
    s32 = float(np.float32(s))
    assert o.b_star == (B * L if s32 / p > B / C0 else 0)
    np.testing.assert_allclose(o.G, [(B + b * s32) / (C0 + p * b) for b in range(B * L + 1)], rtol=1e-14)


@pytest.mark.parametrize("seed", range(10))
def test_slot_price_rule_of_eq_2(orc, seed):
    rng = np.random.default_rng(100 + seed)
    B, L = 16, 15
    S = np.cumprod(rng.uniform(0.6, 1.0, (B, L)), axis=1).astype(np.float32)
    o = orc.size_budget(S, np.full(B, L, np.int32), L, 40.0, 1.0)
    s = np.sort(S.ravel().astype(np.float64))[::-1]
    b = o.b_star
    assert 0 < b < B * L
    lam_prev = o.G[b - 1] * 1.0
    assert s[b - 1] > lam_prev           # the last slot taken raised goodput
    assert s[b] <= o.lam + 1e-15         # the next one would not: s <= lambda = G(b*) p
    assert o.lam == pytest.approx(o.G[b] * 1.0, rel=1e-15)


def test_costlier_slots_shrink_the_budget(orc):
    rng = np.random.default_rng(7)
    S = np.cumprod(rng.uniform(0.5, 1.0, (32, 15)), axis=1).astype(np.float32)
    bs = [orc.size_budget(S, np.full(32, 15, np.int32), 15, 50.0, p).b_star for p in (0.1, 0.3, 1.0, 3.0, 10.0)]
    assert bs == sorted(bs, reverse=True) and bs[0] > bs[-1]


def test_only_verifiable_slots_count(orc):
    rng = np.random.default_rng(8)
    S = np.cumprod(rng.uniform(0.5, 1.0, (8, 15)), axis=1).astype(np.float32)
    chain_len = rng.integers(0, 16, 8).astype(np.int32)
    a = orc.size_budget(S, chain_len, 10, 20.0, 0.5)
    S2 = S.copy()
    for r in range(8):
        S2[r, min(chain_len[r], 10):] = 1.0  # slots past chain_len or max_verify_len
    b = orc.size_budget(S2, chain_len, 10, 20.0, 0.5)
    assert (a.b_star, a.lam) == (b.b_star, b.lam)
    assert len(a.G) == int(np.minimum(chain_len, 10).sum()) + 1
