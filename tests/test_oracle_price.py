"""Pins of the oracle's pricing and allocation (Hybrid Spark sec. 4.2 Eq. (1),
sec. 4.3 Eq. (3), the contains rule, sec. 4.4 / sec. 2 allocation, App. E and
App. G worked numbers, App. H policies)."""
import itertools

import numpy as np
import pytest

import workloads as W


def _logit(p):
    return float(np.log(p / (1 - p)))


# ---------------------------------------------------------------- Eq. (1) pins
def test_shared_intercept_predicts_0_893(orc):
    # App. E: one intercept beta = 2.117 predicts 0.893 at every position
    coef = W.table7_coef(1)
    for k in (1, 7, 15):
        assert round(float(orc.estimate_h(coef, k, 9, 0, 9)), 3) == 0.893


def test_per_position_intercepts_rise_from_0_76_to_0_95(orc):
    # App. E: estimator 2's intercepts 1.158 -> 3.046 are acceptances 0.76 -> 0.95
    coef = W.table7_coef(2)
    assert round(float(orc.estimate_h(coef, 1, 7, 1, 7)), 2) == 0.76
    assert round(float(orc.estimate_h(coef, 15, 7, 1, 7)), 2) == 0.95


def test_copy_length_term_adds_5_7_logits_at_the_first_position(orc):
    # App. D: a 256-token copy adds kappa_first ln(256/15) ~ 5.7 logits to the first
    # position of a full match (Qwen3-4B, Table 5)
    coef = W.table5_coef("qwen3_4b")
    l256 = _logit(float(orc.estimate_h(coef, 1, 15, 1, 256)))
    l15 = _logit(float(orc.estimate_h(coef, 1, 15, 1, 15)))
    assert abs((l256 - l15) - 5.7) < 0.05
    # later positions use kappa_rest
    r256 = _logit(float(orc.estimate_h(coef, 2, 15, 1, 256)))
    r15 = _logit(float(orc.estimate_h(coef, 2, 15, 1, 15)))
    assert abs((r256 - r15) - 1.8333 * np.log(256 / 15)) < 0.01
    # copies beyond the cap add nothing more
    assert orc.estimate_h(coef, 1, 15, 1, 5000) == orc.estimate_h(coef, 1, 15, 1, 256)


def test_full_match_indicator_and_agreement_terms(orc):
    coef = W.table5_coef("qwen3_4b")
    # below a full match, copy length does not enter
    assert orc.estimate_h(coef, 3, 14, 1, 14) == orc.estimate_h(coef, 3, 14, 1, 200)
    # agreement adds delta = 1.2455 logits
    d = _logit(float(orc.estimate_h(coef, 4, 9, 1, 9))) - _logit(float(orc.estimate_h(coef, 4, 9, 0, 9)))
    assert abs(d - 1.2455) < 2e-3
    # match length: w_first per token of (n - 5) at the first position
    w = _logit(float(orc.estimate_h(coef, 1, 10, 0, 10))) - _logit(float(orc.estimate_h(coef, 1, 5, 0, 5)))
    assert abs(w - 5 * -0.0893) < 2e-3
    # the value is the fp32 rounding of the double sigma
    z = -0.220 + 1.2455 + 1.1998 + 2.0118 * np.log(256 / 15) + -0.0893 * 10
    assert orc.estimate_h(coef, 1, 15, 1, 256) == np.float32(1 / (1 + np.exp(-z)))


# ---------------------------------------------------------------- Eq. (3) pins
def test_table8_chain_values(orc):
    # App. G Table 8 (lambda = 0.309): n-gram chain sum S = 5.87 over 15 slots of which
    # 9 exceed lambda with sum 4.35 -> V = 1.57; DSpark's 7 slots sum to 5.58 -> V = 3.42
    lam = 0.309
    above = np.linspace(0.62, 0.346666, 9)
    above *= 4.35 / above.sum()
    below = np.linspace(0.30, 0.2066666, 6)
    below *= 1.52 / below.sum()
    Sg = np.concatenate([above, below]).astype(np.float32)
    Sd = np.linspace(0.95, 0.644, 7)
    Sd = (Sd * 5.58 / Sd.sum()).astype(np.float32)
    assert np.all(np.diff(Sg) <= 0) and np.all(Sg[:9] > lam) and np.all(Sg[9:] < lam)
    assert abs(Sg.sum() - 5.87) < 1e-3 and abs(Sd.sum() - 5.58) < 1e-3
    Vg = float(orc.chain_value(Sg, lam))
    Vd = float(orc.chain_value(Sd, lam))
    assert round(Vg, 2) == 1.57 and round(Vd, 2) == 3.42
    # sum S prefers the n-gram chain, V prefers DSpark's
    assert Sg.sum() > Sd.sum() and Vd > Vg


# ---------------------------------------------------------------- chain choice
def _price(orc, d, c, g, feats, lam=0.04, budget=100, mvl=15, policy="proposed", greedy=True,
           coef=None):
    d = np.atleast_2d(np.asarray(d, np.int32))
    c = np.atleast_2d(np.asarray(c, np.float32))
    B, K = d.shape
    L = 15
    gg = np.full((B, L), -1, np.int32)
    gl = np.zeros(B, np.int32)
    for r, row in enumerate(g if (g and isinstance(g[0], (list, tuple))) else [g]):
        gg[r, :len(row)] = row
        gl[r] = len(row)
    n, a, m = (np.asarray([f[i] for f in (feats if isinstance(feats[0], tuple) else [feats])], np.int32)
               for i in range(3))
    return orc.price_and_allocate(d, c, np.full(B, K, np.int32), gg, gl, n, a, m,
                                  coef or W.table5_coef(), lam, budget, mvl, policy, greedy)


def test_contains_rule_merges_survivals_and_continues_with_h(orc):
    d = [1, 2, 3, 4, 5, 6, 7]
    c = [0.99] * 7
    g = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10]
    out = _price(orc, d, c, g, (15, 1, 40))
    assert out.source[0] == orc.SRC_CONTAINS and out.chain_len[0] == 10
    assert out.chain[0, :10].tolist() == g
    coef = W.table5_coef()
    h = [orc.estimate_h(coef, k, 15, 1, 40) for k in range(1, 11)]
    Sg = np.cumprod(np.array(h, np.float32), dtype=np.float32)
    Sd = np.cumprod(np.array(c, np.float32), dtype=np.float32)
    S = out.S[0]
    for k in range(7):
        assert S[k] == max(Sg[k], Sd[k])
    for k in range(7, 10):
        assert S[k] == np.float32(S[k - 1] * h[k])
    assert np.all(out.point_mass[0, :10] == 1)


def test_value_rule_ties_go_to_the_ngram_chain(orc):
    # both chains entirely below the price: V^g = V^d = 0 -> the n-gram chain
    out = _price(orc, [1] * 7, [0.1] * 7, [9, 9, 9], (5, 0, 5), lam=0.99)
    assert out.source[0] == orc.SRC_NGRAM
    # no match: the model chain
    out = _price(orc, [1] * 7, [0.9] * 7, [], (0, 0, 0))
    assert out.source[0] == orc.SRC_MODEL and out.chain_len[0] == 7


def test_value_rule_prefers_the_higher_value(orc):
    weak = (5, 0, 5)  # short match, runner-up disagrees: low h
    out = _price(orc, [1] * 7, [0.95] * 7, list(range(20, 35)), weak, lam=0.3)
    assert out.source[0] == orc.SRC_MODEL
    strong = (15, 1, 256)
    out = _price(orc, [1] * 7, [0.6] * 7, list(range(20, 35)), strong, lam=0.3)
    assert out.source[0] == orc.SRC_NGRAM


def test_policies(orc):
    d = [1, 2, 3, 4, 5, 6, 7]
    g_ext = d + [8, 9, 10]
    out = _price(orc, d, [0.99] * 7, [40, 41], (5, 0, 5), policy="ngram_first")
    assert out.source[0] == orc.SRC_NGRAM and out.chain_len[0] == 2
    out = _price(orc, d, [0.99] * 7, [], (0, 0, 0), policy="ngram_first")
    assert out.source[0] == orc.SRC_MODEL
    out = _price(orc, d, [0.9] * 7, g_ext, (15, 1, 100), policy="extension", greedy=False)
    assert out.source[0] == orc.SRC_EXTENSION and out.chain_len[0] == 10
    Sd = np.cumprod(np.array([0.9] * 7, np.float32), dtype=np.float32)
    assert np.array_equal(out.S[0, :7], Sd)
    # the tail continues from S^d_7 and never outranks the model's own slots
    assert np.all(out.S[0, 7:10] <= out.S[0, 6])
    assert out.point_mass[0, :7].tolist() == [0] * 7 and out.point_mass[0, 7:10].tolist() == [1] * 3
    out = _price(orc, d, [0.9] * 7, [1, 2, 9, 9, 9, 9, 9, 9], (15, 1, 100), policy="extension")
    assert out.source[0] == orc.SRC_MODEL and out.chain_len[0] == 7
    out = _price(orc, d, [0.9] * 7, [5, 6], (5, 1, 5), policy="model_only")
    assert out.source[0] == orc.SRC_MODEL
    out = _price(orc, d, [0.9] * 7, [5, 6], (5, 1, 5), policy="ngram_only")
    assert out.source[0] == orc.SRC_NGRAM and out.chain_len[0] == 2
    # probabilistic model tokens are not point masses; n-gram tokens always are
    out = _price(orc, d, [0.99] * 7, [], (0, 0, 0), greedy=False)
    assert out.point_mass[0, :7].tolist() == [0] * 7


def test_confidences_outside_unit_interval_are_clamped_and_flagged(orc):
    out = _price(orc, [1] * 7, [1.5, 0.9, -0.1, 0.9, 0.9, 0.9, 0.9], [], (0, 0, 0))
    assert out.status & orc.ST_BAD_VALUE
    assert out.S[0, 0] == 1.0 and out.S[0, 2] == 0.0


# ---------------------------------------------------------------- allocation
def test_allocation_is_the_best_prefix_closed_set_brute_force(orc):
    rng = np.random.default_rng(3)
    for trial in range(300):
        B = int(rng.integers(1, 4))
        K = 4
        cvals = rng.choice([0.5, 0.7, 0.8, 0.9, 1.0], (B, K)).astype(np.float32)
        d = rng.integers(0, 50, (B, K)).astype(np.int32)
        d_len = rng.integers(0, K + 1, B).astype(np.int32)
        L = 4
        g = np.full((B, L), -1, np.int32)
        budget = int(rng.integers(0, 12))
        mvl = int(rng.integers(0, 5))
        out = orc.price_and_allocate(d, cvals, d_len, g, np.zeros(B, np.int32), np.zeros(B, np.int32),
                                     np.zeros(B, np.int32), np.zeros(B, np.int32), W.table5_coef(),
                                     0.1, budget, mvl, "model_only", True)
        caps = [min(int(out.chain_len[r]), mvl) for r in range(B)]
        total = min(budget, sum(caps))
        S = out.S.astype(np.float64)
        best = None
        for alloc in itertools.product(*[range(cp + 1) for cp in caps]):
            if sum(alloc) != total:
                continue
            val = sum(S[r, :alloc[r]].sum() for r in range(B))
            key = (val,)
            if best is None or val > best[0] + 1e-12:
                best = (val, alloc)
        got = tuple(int(v) for v in out.verify_len)
        assert sum(got) == total
        got_val = sum(S[r, :got[r]].sum() for r in range(B))
        assert got_val >= best[0] - 1e-9, (got, best)
        assert out.row_off.tolist() == np.concatenate([[0], np.cumsum(np.asarray(got) + 1)]).tolist()


def test_allocation_ties_go_to_lower_request_then_position(orc):
    B, K = 3, 4
    c = np.full((B, K), 1.0, np.float32)  # every slot has S = 1
    out = orc.price_and_allocate(np.zeros((B, K), np.int32), c, np.full(B, K, np.int32),
                                 np.full((B, 4), -1, np.int32), np.zeros(B, np.int32),
                                 np.zeros(B, np.int32), np.zeros(B, np.int32), np.zeros(B, np.int32),
                                 W.table5_coef(), 0.1, 6, 4, "model_only", True)
    assert out.verify_len.tolist() == [4, 2, 0]


def test_price_does_not_gate_allocation(orc):
    # lambda acts in the chain choice only: slots below it are still allocated
    out = _price(orc, [1] * 7, [0.5] * 7, [], (0, 0, 0), lam=0.9, budget=5)
    assert out.verify_len[0] == 5


def test_contains_rule_dominance_on_enumerated_greedy_targets(orc):
    # sec. 4.3: an n-gram chain that starts with all of d is accepted at least as far
    # as d on every target draw.  Enumerate greedy targets over a 3-token vocabulary.
    V, K = 3, 2
    d = [1, 2]
    for gtail in itertools.product(range(V), repeat=2):
        g = d + list(gtail)
        for argmaxes in itertools.product(range(V), repeat=len(g) + 1):
            rows = np.full((len(g) + 1, V), -1.0, np.float32)
            rows[np.arange(len(g) + 1), argmaxes] = 1.0
            acc = []
            for chain in (g, d):
                ch = np.full((1, 15), -1, np.int32)
                ch[0, :len(chain)] = chain
                ro = np.array([0, len(g) + 1], np.int32)
                out = orc.verify_chain(rows, ro, ch, np.array([len(chain)], np.int32))
                acc.append(int(out.n_accepted[0]))
            assert acc[0] >= acc[1]
