"""Pins of the oracle's candidate-tree builder (AdaSpark sec. 2.2 tree shape,
sec. 3.1 Proposition 1 best-first order, sec. 3.3 Eq. (6) and n-gram
candidates, Algorithm 1 depth-first layout).

Closed forms: a chain-only tree is a path whose q are logistic sigmoids; a
parent whose m children share one score gives each e^s / (1 + m e^s).  Brute
force: on small blocks, no tree of width - 1 candidates has a larger sum of Q
than the built one (Proposition 1), and every prefix of the order is a tree.
Merge rules, ties and the layout are checked on hand-built blocks."""
import itertools
import math

import numpy as np
import pytest


def f32(x):
    """the fp32 value the builder receives for a score"""
    return float(np.float32(x))


def _block(rng, P, Kc, V=50):
    tok = np.stack([rng.choice(V, Kc, replace=False) for _ in range(P)])[None].astype(np.int32)
    score = rng.normal(0, 1.5, (1, P, Kc)).astype(np.float32)
    return tok, score


def _tree_of(o, r=0):
    """candidate id of every row and the parent candidate id"""
    n = int(o.n_rows[r])
    cid = o.cand_id[r, :n]
    par = [-1 if o.parent[r, j] < 0 else int(cid[o.parent[r, j]]) for j in range(n)]
    return list(map(int, cid)), par


def test_chain_only_tree_is_a_path_of_sigmoids(orc):
    s = 0.7
    Lg = 6
    o = orc.build_tree([3], np.zeros((1, 0, 1), np.int32), np.zeros((1, 0, 1), np.float32),
                       [np.arange(100, 100 + Lg)], [Lg], [s], [0.0], 10)
    sig = 1.0 / (1.0 + math.exp(-f32(s)))
    assert o.n_rows[0] == 1 + Lg
    np.testing.assert_allclose(o.Q[0, 1:1 + Lg], [sig ** k for k in range(1, Lg + 1)], rtol=1e-13)
    assert list(o.parent[0, :1 + Lg]) == [-1] + list(range(Lg))
    assert list(o.tok[0, :1 + Lg]) == [3] + list(range(100, 100 + Lg))


@pytest.mark.parametrize("m,s", [(1, 0.0), (4, -1.3), (8, 2.0)])
def test_equal_scores_share_one_softmax_with_none(orc, m, s):
    tok = np.arange(m, dtype=np.int32).reshape(1, 1, m)
    o = orc.build_tree([99], tok, np.full((1, 1, m), s, np.float32), np.zeros((1, 1), np.int32), [0], [0.0],
                       [0.0], m + 1)
    want = math.exp(f32(s)) / (1.0 + m * math.exp(f32(s)))
    np.testing.assert_allclose(o.Q[0, 1:1 + m], want, rtol=1e-14)
    assert o.Q[0, 1:1 + m].sum() < 1.0  # the "none" outcome keeps the rest


def test_picks_form_a_spine_and_siblings_are_leaves(orc):
    P, Kc = 4, 3  # the shape of the page's Figure 1
    tok = (10 * np.arange(1, P + 1)[:, None] + np.arange(Kc)[None]).astype(np.int32)[None]
    score = np.where(np.arange(Kc)[None] == 0, 3.0, -1.0).astype(np.float32)[None].repeat(P, 1)
    o = orc.build_tree([1], tok, score, np.zeros((1, 1), np.int32), [0], [0.0], [0.0], 1 + P * Kc)
    cid, par = _tree_of(o)
    pc = dict(zip(cid, par))
    for i in range(P):
        pick = 1 + i * Kc
        assert pc[pick] == (0 if i == 0 else 1 + (i - 1) * Kc)
        for k in range(1, Kc):
            assert pc[pick + k] == pc[pick]  # a sibling hangs from the pick's parent
            assert (pick + k) not in pc.values()  # and has no children


def test_ngram_chain_agrees_with_picks_then_extends(orc):
    P, Kc, adj = 2, 3, 1.5
    tok = np.array([[[10, 11, 12], [20, 21, 22]]], np.int32)
    score = np.zeros((1, P, Kc), np.float32)
    o = orc.build_tree([5], tok, score, [[10, 20, 30, 40]], [4], [0.4], [adj], 16)
    # no node for 10 and 20 (agreed picks); 30 and 40 are n-gram nodes under pick 1
    cid, par = _tree_of(o)
    assert o.n_rows[0] == 1 + P * Kc + 2
    pc = dict(zip(cid, par))
    assert pc[7] == 4 and pc[8] == 7
    e = math.exp
    den = 1 + e(adj) + 2 * e(-adj)  # agreed pick +adj, contradicted siblings -adj
    np.testing.assert_allclose(o.Q[0, 1], e(adj) / den, rtol=1e-13)
    np.testing.assert_allclose(o.Q[0, 2], e(-adj) / den, rtol=1e-13)
    sig = 1 / (1 + e(-f32(0.4)))
    np.testing.assert_allclose(o.Q[0, 8], o.Q[0, 4] * sig * sig, rtol=1e-13)


def test_ngram_chain_that_matches_no_candidate_contradicts_them_all(orc):
    P, Kc, adj, sg = 2, 2, f32(0.8), -0.5
    tok = np.array([[[10, 11], [20, 21]]], np.int32)
    o = orc.build_tree([5], tok, np.zeros((1, P, Kc), np.float32), [[77, 78]], [2], [sg], [adj], 16)
    e = math.exp
    den = 1 + 2 * e(-adj) + e(sg)  # both position-0 candidates contradicted, one n-gram child
    np.testing.assert_allclose(o.Q[0, 1], e(-adj) / den, rtol=1e-13)
    np.testing.assert_allclose(o.Q[0, 5], e(sg) / den, rtol=1e-13)
    cid, par = _tree_of(o)
    assert dict(zip(cid, par))[6] == 5


def test_ngram_chain_through_a_sibling_continues_below_it(orc):
    tok = np.array([[[10, 11, 12], [20, 21, 22]]], np.int32)
    o = orc.build_tree([5], tok, np.zeros((1, 2, 3), np.float32), [[12, 50]], [2], [0.0], [0.0], 16)
    cid, par = _tree_of(o)
    assert dict(zip(cid, par))[7] == 3  # the n-gram node hangs from the agreed sibling


def test_ties_go_to_the_lower_index(orc):
    Kc = 6
    tok = np.arange(Kc, dtype=np.int32).reshape(1, 1, Kc)
    o = orc.build_tree([0], tok, np.zeros((1, 1, Kc), np.float32), np.zeros((1, 1), np.int32), [0], [0.0],
                       [0.0], 4)
    cid, _ = _tree_of(o)
    assert sorted(cid) == [0, 1, 2, 3]


def _random_case(rng, P, Kc, Lg):
    tok, score = _block(rng, P, Kc)
    chain = []
    cur_pos = 0
    for t in range(Lg):  # follow the picks for a while, then leave the block
        if cur_pos < P and rng.random() < 0.6:
            chain.append(int(tok[0, cur_pos, 0] if rng.random() < 0.8 else tok[0, cur_pos, 1]))
            cur_pos += 1
        else:
            chain.append(int(rng.integers(1000, 2000)))
            cur_pos = P
    return tok, score, np.array([chain], np.int32), [float(rng.normal(0, 1))], [float(abs(rng.normal(0, 1)))]


@pytest.mark.parametrize("seed", range(12))
def test_proposition_1_by_brute_force(orc, seed):
    rng = np.random.default_rng(seed)
    P, Kc, Lg = 2, 3, 3
    tok, score, chain, sg, adj = _random_case(rng, P, Kc, Lg)
    full = orc.build_tree([0], tok, score, chain, [Lg], sg, adj, 64)
    N = int((full.Q[0] >= 0).sum())
    cid_full, par_full = _tree_of(full)
    cpar = dict(zip(cid_full, par_full))
    Q = full.Q[0, :N]
    for width in range(2, N + 1):
        o = orc.build_tree([0], tok, score, chain, [Lg], sg, adj, width)
        cid, par = _tree_of(o)
        got = set(cid) - {0}
        assert all(cpar[c] in got | {0} for c in got)  # a tree
        best = max(sum(Q[list(sub)]) for sub in itertools.combinations(range(1, N), width - 1)
                   if all(cpar[c] in set(sub) | {0} for c in sub))
        assert sum(Q[list(got)]) >= best - 1e-15
        if width > 2:  # the order's prefixes are nested
            assert prev <= got
        prev = got


@pytest.mark.parametrize("seed", range(6))
def test_layout_is_depth_first_with_children_in_index_order(orc, seed):
    rng = np.random.default_rng(100 + seed)
    P, Kc, Lg = 5, 4, 8
    tok, score, chain, sg, adj = _random_case(rng, P, Kc, Lg)
    o = orc.build_tree([0], tok, score, chain, [Lg], sg, adj, 14)
    n = int(o.n_rows[0])
    par = o.parent[0, :n]
    cid = o.cand_id[0, :n]
    assert par[0] == -1 and all(0 <= par[j] < j for j in range(1, n))
    # preorder: each subtree is one contiguous block of rows
    for j in range(n):
        sub = {j}
        for k in range(j + 1, n):
            if par[k] in sub:
                sub.add(k)
        assert sub == set(range(j, j + len(sub)))
    # siblings appear in increasing candidate index
    for j in range(n):
        kids = [k for k in range(n) if par[k] == j]
        assert list(cid[kids]) == sorted(cid[kids])
    assert np.all(o.tok[0, n:] == -1) and np.all(o.cand_id[0, n:] == -1)


# ------------------------------------------------------------------ chains from the anchor and each pick
def _chains(rows, Lg):
    """[C x Lg] chain tokens (padded with -1) and their lengths"""
    tok = np.full((1, len(rows), Lg), -1, np.int32)
    for c, r in enumerate(rows):
        tok[0, c, :len(r)] = r
    return tok, np.array([[len(r) for r in rows]], np.int32)


def test_chains_from_picks_share_their_nodes(orc):
    # picks 10, 20 with siblings 11, 21.  Chain 0 agrees with both picks and adds
    # 30; chain 1 (from pick 0) walks the same way and adds 40 below 30; chain 2
    # (from pick 1) reuses 30 and adds 50 beside 40
    tok = np.array([[[10, 11], [20, 21]]], np.int32)
    ng, ln = _chains([[10, 20, 30], [20, 30, 40], [30, 50]], 4)
    o = orc.build_tree([5], tok, np.zeros((1, 2, 2), np.float32), ng, ln, [0.0], [0.0], 32)
    assert int((o.Q[0] >= 0).sum()) == 1 + 4 + 3
    cid, par = _tree_of(o)
    pc = dict(zip(cid, par))
    assert pc[5] == 3 and pc[6] == 5 and pc[7] == 5
    # 30 has two children, both n-gram nodes with score 0: e^0 / (1 + 2 e^0) each
    np.testing.assert_allclose(o.Q[0, 6] / o.Q[0, 5], 1.0 / 3.0, rtol=1e-14)


def test_a_candidate_agreed_by_one_chain_and_contradicted_by_another_is_agreed(orc):
    adj = f32(0.9)
    tok = np.array([[[10, 11], [20, 21]]], np.int32)
    # chain 0: pick 10, then sibling 21 (20 contradicted); chain 1 from pick 0: 20 (21 contradicted)
    ng, ln = _chains([[10, 21], [20]], 2)
    o = orc.build_tree([5], tok, np.zeros((1, 2, 2), np.float32), ng, ln, [0.0], [adj], 16)
    e = math.exp
    q0 = e(adj) / (1 + e(adj) + e(-adj))  # pick 10 agreed, sibling 11 contradicted
    np.testing.assert_allclose(o.Q[0, 1], q0, rtol=1e-13)
    np.testing.assert_allclose(o.Q[0, 3], q0 * e(adj) / (1 + 2 * e(adj)), rtol=1e-13)
    np.testing.assert_allclose(o.Q[0, 4], q0 * e(adj) / (1 + 2 * e(adj)), rtol=1e-13)


def test_one_chain_in_the_chain_layout_equals_the_single_chain_call(orc):
    rng = np.random.default_rng(5)
    tok, score, chain, sg, adj = _random_case(rng, 4, 3, 6)
    a = orc.build_tree([0], tok, score, chain, [6], sg, adj, 12)
    b = orc.build_tree([0], tok, score, chain[:, None, :], [[6]], sg, adj, 12)
    for f in ("tok", "parent", "cand_id", "n_rows"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    np.testing.assert_array_equal(a.Q, b.Q)


def _random_chains(rng, tok, P, Lg):
    rows = []
    for c in range(P + 1):
        r, pos = [], c
        for _ in range(int(rng.integers(0, Lg + 1))):
            if pos < P and rng.random() < 0.6:
                r.append(int(tok[0, pos, int(rng.integers(0, tok.shape[2]))]))
                pos += 1
            else:
                r.append(int(rng.integers(1000, 1004)))  # few values: chains meet again
                pos = P
        rows.append(r)
    return _chains(rows, Lg)


@pytest.mark.parametrize("seed", range(10))
def test_proposition_1_by_brute_force_with_chains_from_every_pick(orc, seed):
    rng = np.random.default_rng(200 + seed)
    P, Kc, Lg = 2, 2, 2
    tok, score = _block(rng, P, Kc)
    ng, ln = _random_chains(rng, tok, P, Lg)
    sg, adj = [float(rng.normal(0, 1))], [float(abs(rng.normal(0, 1)))]
    full = orc.build_tree([0], tok, score, ng, ln, sg, adj, 64)
    N = int((full.Q[0] >= 0).sum())
    cid_full, par_full = _tree_of(full)
    cpar = dict(zip(cid_full, par_full))
    assert sorted(cid_full) == list(range(N))
    Q = full.Q[0, :N]
    prev = None
    for width in range(2, min(N, 9) + 1):
        o = orc.build_tree([0], tok, score, ng, ln, sg, adj, width)
        got = set(_tree_of(o)[0]) - {0}
        assert all(cpar[c] in got | {0} for c in got)
        best = max(sum(Q[list(sub)]) for sub in itertools.combinations(range(1, N), width - 1)
                   if all(cpar[c] in set(sub) | {0} for c in sub))
        assert sum(Q[list(got)]) >= best - 1e-15
        if prev is not None:
            assert prev <= got
        prev = got


@pytest.mark.parametrize("seed", range(4))
def test_layout_with_chains_from_every_pick(orc, seed):
    rng = np.random.default_rng(300 + seed)
    P, Kc, Lg = 5, 3, 6
    tok, score = _block(rng, P, Kc)
    ng, ln = _random_chains(rng, tok, P, Lg)
    o = orc.build_tree([0], tok, score, ng, ln, [0.3], [0.5], 20)
    n = int(o.n_rows[0])
    par, cid = o.parent[0, :n], o.cand_id[0, :n]
    assert par[0] == -1 and all(0 <= par[j] < j for j in range(1, n))
    for j in range(n):
        kids = [k for k in range(n) if par[k] == j]
        assert list(cid[kids]) == sorted(cid[kids])
        assert len({int(o.tok[0, k]) for k in kids if cid[k] > P * Kc}) == \
            len([k for k in kids if cid[k] > P * Kc])  # n-gram children carry distinct tokens
