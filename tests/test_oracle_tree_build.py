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
