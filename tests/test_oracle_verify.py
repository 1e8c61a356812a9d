"""Pins of the oracle's chain verification (Hybrid Spark sec. 2 and App. H;
the fixed-cost parallel drafter page's accept / resample rule, under which a
round that accepts r drafts emits r + 1 tokens).

The central pin is exact losslessness: on tiny vocabularies the law of the
tokens a round emits, continued by the target itself, equals the target's own
law, for probabilistic drafts and for point masses.  The oracle is treated as
a black box: its decision regions in (u_i, u'_i) are located by bisection on
its outputs, so the check does not restate its formulas."""
import itertools

import numpy as np
import pytest


def _softmax(z, T):
    z = np.asarray(z, np.float64) / T
    z = z - z.max()
    p = np.exp(z)
    return p / p.sum()


class _Tables:
    """Prefix-dependent logits of a tiny target and drafter."""

    def __init__(self, V, seed, scale=1.5):
        self.V, self.rng, self.scale = V, np.random.default_rng(seed), scale
        self.t, self.d = {}, {}

    def target(self, prefix):
        key = tuple(prefix)
        if key not in self.t:
            self.t[key] = (self.rng.standard_normal(self.V) * self.scale).astype(np.float32)
        return self.t[key]

    def draft(self, prefix):
        key = tuple(prefix)
        if key not in self.d:
            self.d[key] = (self.rng.standard_normal(self.V) * self.scale).astype(np.float32)
        return self.d[key]


def _run(orc, tab, y, use_q, T, u):
    ell = len(y)
    V = tab.V
    L = max(ell, 1)
    rows = np.stack([tab.target(y[:i]) for i in range(ell + 1)]).astype(np.float32)
    ch = np.full((1, L), -1, np.int32)
    ch[0, :ell] = y
    pm = np.ones((1, L), np.uint8)
    draft = None
    if use_q:
        pm[0, :ell] = 0
        draft = np.zeros((1, max(ell, 1), V), np.float32)
        for i in range(ell):
            draft[0, i] = tab.draft(y[:i])
    uo = np.zeros((1, L + 1, 2))
    uo[0, :len(u)] = u
    out = orc.verify_chain(rows, np.array([0, ell + 1], np.int32), ch, np.array([ell], np.int32),
                           pm, draft, temperature=T, u_override=uo)
    n = int(out.n_emitted[0])
    return tuple(int(v) for v in out.out_tokens[0, :n]), int(out.n_accepted[0])


def _bisect(pred, lo=0.0, hi=1.0, iters=60):
    """sup{x in [lo, hi): pred(x)} for a predicate true on [lo, a) and false after."""
    if not pred(lo):
        return lo
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return hi


def _round_law(orc, tab, y, use_q, T):
    """{emitted tuple: probability} of one round, located by bisection on the oracle."""
    V, ell = tab.V, len(y)
    law = {}

    def token_law(i, base):
        # out token at position i as u'_i sweeps [0, 1): boundaries by bisection
        def tok_at(x):
            u = [list(p) for p in base]
            u[i - 1][1] = x
            return _run(orc, tab, y, use_q, T, u)[0]

        res = {}
        prev = 0.0
        for x in range(V):
            b = _bisect(lambda v: tok_at(v)[i - 1] <= x) if x < V - 1 else 1.0
            if b > prev:
                res[tok_at(0.5 * (prev + b))] = res.get(tok_at(0.5 * (prev + b)), 0.0) + (b - prev)
            prev = max(prev, b)
        return res

    def walk(i, base, weight):
        if i == ell + 1:  # every draft accepted: the bonus draw
            for seq, w in token_law(i, base).items():
                law[seq] = law.get(seq, 0.0) + weight * w
            return

        def accepted(x):
            u = [list(p) for p in base]
            u[i - 1][0] = x
            return _run(orc, tab, y, use_q, T, u)[1] >= i

        a = _bisect(accepted)
        if a > 0:
            nb = [list(p) for p in base]
            nb[i - 1][0] = 0.5 * a
            walk(i + 1, nb, weight * a)
        if a < 1:
            nb = [list(p) for p in base]
            nb[i - 1][0] = 0.5 * (a + 1.0)
            for seq, w in token_law(i, nb).items():
                law[seq] = law.get(seq, 0.0) + weight * (1.0 - a) * w

    walk(1, [[0.0, 0.0] for _ in range(ell + 1)], 1.0)
    return law


def _extend(tab, law, H, T):
    """continue every emitted prefix with the target itself up to H tokens"""
    out = {}
    for seq, w in law.items():
        stack = [(seq, w)]
        while stack:
            s, ws = stack.pop()
            if len(s) == H:
                out[s] = out.get(s, 0.0) + ws
                continue
            p = _softmax(tab.target(s), T)
            for x in range(tab.V):
                stack.append((s + (x,), ws * p[x]))
    return out


def _target_law(tab, H, T):
    law = {}
    for s in itertools.product(range(tab.V), repeat=H):
        w = 1.0
        for k in range(H):
            w *= _softmax(tab.target(s[:k]), T)[s[k]]
        law[s] = w
    return law


@pytest.mark.parametrize("V,ell,T,seed", [(3, 1, 1.0, 0), (3, 2, 0.7, 1), (4, 2, 1.0, 2), (3, 3, 1.3, 3)])
def test_lossless_with_probabilistic_drafts(orc, V, ell, T, seed):
    tab = _Tables(V, seed)
    total = {}
    for y in itertools.product(range(V), repeat=ell):
        wq = 1.0
        for i in range(ell):
            wq *= _softmax(tab.draft(y[:i]), T)[y[i]]
        for s, w in _extend(tab, _round_law(orc, tab, list(y), True, T), ell + 1, T).items():
            total[s] = total.get(s, 0.0) + wq * w
    want = _target_law(tab, ell + 1, T)
    assert abs(sum(total.values()) - 1.0) < 1e-9
    for s in want:
        assert abs(total.get(s, 0.0) - want[s]) < 1e-9, s


@pytest.mark.parametrize("V,ell,T,seed", [(3, 2, 1.0, 4), (4, 3, 0.7, 5)])
def test_lossless_with_point_mass_drafts(orc, V, ell, T, seed):
    tab = _Tables(V, seed)
    want = _target_law(tab, ell + 1, T)
    for y in itertools.product(range(V), repeat=ell):  # every fixed chain on its own
        got = _extend(tab, _round_law(orc, tab, list(y), False, T), ell + 1, T)
        for s in want:
            assert abs(got.get(s, 0.0) - want[s]) < 1e-9, (y, s)


def test_r_accepted_emit_r_plus_one(orc):
    rng = np.random.default_rng(9)
    B, V, L, K = 16, 50, 6, 4
    ell = rng.integers(0, L + 1, B).astype(np.int32)
    row_off = np.concatenate([[0], np.cumsum(ell + 1)]).astype(np.int32)
    logits = rng.standard_normal((row_off[-1], V)).astype(np.float32)
    chain = rng.integers(0, V, (B, L)).astype(np.int32)
    draft = rng.standard_normal((B, K, V)).astype(np.float32)
    pm = (rng.random((B, L)) < 0.5).astype(np.uint8)
    pm[:, K:] = 1
    for T in (0.0, 0.5, 1.0):
        for step in range(5):
            out = orc.verify_chain(logits, row_off, chain, ell, pm, draft, T, 1, step)
            assert np.all(out.n_emitted == out.n_accepted + 1)
            assert np.all(out.n_accepted <= ell)
            for r in range(B):
                n = out.n_accepted[r]
                assert out.out_tokens[r, :n].tolist() == chain[r, :n].tolist()
                assert np.all(out.out_tokens[r, n + 1:] == -1)
                assert 0 <= out.out_tokens[r, n] < V


def test_greedy_is_the_longest_argmax_matching_prefix(orc):
    rng = np.random.default_rng(11)
    B, V, L = 32, 20, 7
    ell = rng.integers(0, L + 1, B).astype(np.int32)
    row_off = np.concatenate([[0], np.cumsum(ell + 1)]).astype(np.int32)
    logits = rng.standard_normal((row_off[-1], V)).astype(np.float32)
    am = logits.argmax(axis=1)
    chain = rng.integers(0, V, (B, L)).astype(np.int32)
    for r in range(B):  # make a random number of leading drafts right
        k = int(rng.integers(0, ell[r] + 1))
        chain[r, :k] = am[row_off[r]:row_off[r] + k]
    out = orc.verify_chain(logits, row_off, chain, ell)
    for r in range(B):
        n = 0
        while n < ell[r] and chain[r, n] == am[row_off[r] + n]:
            n += 1
        assert out.n_accepted[r] == n
        assert out.out_tokens[r, n] == am[row_off[r] + n]


def test_greedy_ties_go_to_the_lowest_index(orc):
    row = np.array([[0.5, 2.0, 2.0, -1.0]], np.float32)
    assert orc.row_argmax(row) == 1
    out = orc.verify_chain(row, np.array([0, 1], np.int32), np.full((1, 1), -1, np.int32),
                           np.array([0], np.int32))
    assert out.out_tokens[0, 0] == 1


def test_bonus_draws_follow_p_chi_square(orc):
    # Philox-driven draws over many steps: the bonus token follows p (V = 16)
    V, n = 16, 20000
    rng = np.random.default_rng(12)
    row = (rng.standard_normal((1, V)) * 1.2).astype(np.float32)
    p = _softmax(row[0], 1.0)
    counts = np.zeros(V)
    ch = np.full((1, 1), -1, np.int32)
    for step in range(n):
        out = orc.verify_chain(row, np.array([0, 1], np.int32), ch, np.array([0], np.int32),
                               temperature=1.0, seed=123, step=step)
        counts[out.out_tokens[0, 0]] += 1
    exp = n * p
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 45.0, chi2  # chi2(15) 99.99th percentile ~ 44


def test_point_mass_rejection_draws_follow_p_chi_square(orc):
    # the first emitted token of a one-draft point-mass round follows p_1
    V, n = 8, 20000
    rng = np.random.default_rng(13)
    rows = (rng.standard_normal((2, V)) * 1.0).astype(np.float32)
    p = _softmax(rows[0], 1.0)
    counts = np.zeros(V)
    ch = np.array([[3]], np.int32)
    for step in range(n):
        out = orc.verify_chain(rows, np.array([0, 2], np.int32), ch, np.array([1], np.int32),
                               np.ones((1, 1), np.uint8), temperature=1.0, seed=5, step=step)
        counts[out.out_tokens[0, 0]] += 1
    exp = n * p
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 30.0, chi2  # chi2(7) 99.99th percentile ~ 29.9


def test_residual_row_and_debug_outputs(orc):
    rng = np.random.default_rng(14)
    V, L = 64, 3
    rows = rng.standard_normal((L + 1, V)).astype(np.float32)
    draft = rng.standard_normal((1, L, V)).astype(np.float32)
    ch = rng.integers(0, V, (1, L)).astype(np.int32)
    ro = np.array([0, L + 1], np.int32)
    pm = np.zeros((1, L), np.uint8)
    for step in range(40):
        out = orc.verify_chain(rows, ro, ch, np.array([L], np.int32), pm, draft, 1.0, 2, step)
        i = int(out.pos[0])
        rej = out.n_accepted[0] < L
        w = orc.residual_row(rows, ro, ch, 0, i, rej, pm, draft, 1.0)
        Z = w.sum()
        assert abs(Z - out.Z[0]) < 1e-12
        x = out.out_tokens[0, i - 1]
        cdf = np.cumsum(w)
        assert (cdf[x - 1] if x > 0 else 0.0) <= out.t[0] < cdf[x]
        assert abs(out.resid[0] - w[x] / Z) < 1e-15
        for k in range(1, i + (0 if rej else 1)):
            if k <= L and k < i + 1 and k <= L:
                pk = _softmax(rows[k - 1], 1.0)[ch[0, k - 1]]
                qk = _softmax(draft[0, k - 1], 1.0)[ch[0, k - 1]]
                if k <= i:
                    assert abs(out.ratio[0, k - 1] - pk / qk) < 1e-9 * max(1.0, pk / qk)


def test_bad_layouts_and_tokens_are_flagged(orc):
    V = 10
    rows = np.zeros((4, V), np.float32)
    ch = np.array([[1, 2, 3]], np.int32)
    out = orc.verify_chain(rows, np.array([0, 2], np.int32), ch, np.array([2], np.int32))
    assert out.status & orc.ST_BAD_LENGTH and out.n_emitted[0] == 0
    out = orc.verify_chain(rows, np.array([0, 4], np.int32), np.array([[1, 99, 3]], np.int32),
                           np.array([3], np.int32))
    assert out.status & orc.ST_BAD_TOKEN
    bad = rows.copy()
    bad[1, 3] = np.nan
    out = orc.verify_chain(bad, np.array([0, 4], np.int32), ch, np.array([3], np.int32))
    assert out.status & orc.ST_NONFINITE
