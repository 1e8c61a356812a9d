"""Pins of the oracle's greedy tree verification (AdaSpark sec. 2.2, sec. 3.5)
and of the tree generator's best-first order (AdaSpark sec. 3.1, Prop. 1)."""
import itertools

import numpy as np
import pytest

import workloads as W


def _planted_rows(rng, n, V, want):
    """rows whose argmax is want[j] (or random where want[j] < 0)"""
    rows = rng.standard_normal((n, V)).astype(np.float32)
    for j, t in enumerate(want):
        if t >= 0:
            rows[j, t] += 10.0
    return rows


def test_chain_shaped_tree_equals_greedy_chain_verify(orc):
    # a chain is a tree with one child per node (sec. 2.2); a tree node whose ancestors
    # are a chain's rows computes that chain row (sec. 3.5)
    rng = np.random.default_rng(21)
    V, L = 40, 7
    for trial in range(200):
        ell = int(rng.integers(0, L + 1))
        rows = rng.standard_normal((ell + 1, V)).astype(np.float32)
        am = rows.argmax(1)
        chain = rng.integers(0, V, L).astype(np.int32)
        k = int(rng.integers(0, ell + 1))
        chain[:k] = am[:k]
        cv = orc.verify_chain(rows, np.array([0, ell + 1], np.int32), chain[None, :],
                              np.array([ell], np.int32))
        tok = np.concatenate([[7], chain[:ell]]).astype(np.int32)
        parent = np.arange(-1, ell, dtype=np.int32)
        tv = orc.verify_tree(rows, np.array([0, ell + 1], np.int32), tok, parent, L + 1)
        n = int(cv.n_emitted[0])
        assert tv.accept_len[0] == cv.n_accepted[0]
        assert tv.out_tokens[0, :n].tolist() == cv.out_tokens[0, :n].tolist()
        assert tv.path[0, :n].tolist() == list(range(n))


def _random_tree(rng, n, V, dup=False):
    parent = np.array([-1] + [int(rng.integers(0, j)) for j in range(1, n)], np.int32)
    tok = np.zeros(n, np.int32)
    for j in range(1, n):
        sib = [tok[i] for i in range(1, j) if parent[i] == parent[j]]
        t = int(rng.integers(0, V))
        while not dup and t in sib:
            t = int(rng.integers(0, V))
        tok[j] = t
    return tok, parent


def test_path_by_brute_force_over_root_to_node_paths(orc):
    rng = np.random.default_rng(22)
    V = 6
    for trial in range(400):
        n = int(rng.integers(1, 10))
        tok, parent = _random_tree(rng, n, V, dup=bool(trial % 3 == 0))
        rows = rng.standard_normal((n, V)).astype(np.float32)
        # plant argmaxes that often follow a child
        for j in range(n):
            kids = [c for c in range(n) if parent[c] == j]
            if kids and rng.random() < 0.7:
                rows[j, tok[kids[int(rng.integers(0, len(kids)))]]] += 5
        am = rows.argmax(1)
        # every root-to-node path; a node is reachable iff each step matches the
        # parent's argmax and no lower-index sibling matched first
        def accepted(j):
            while j != 0:
                p = parent[j]
                first = min(c for c in range(n) if parent[c] == p and tok[c] == am[p]) \
                    if any(parent[c] == p and tok[c] == am[p] for c in range(n)) else None
                if first != j:
                    return False
                j = p
            return True
        acc = [j for j in range(n) if accepted(j)]
        deepest = max(acc, key=lambda j: (len(_anc(parent, j)), -j))
        want_path = _anc(parent, deepest)[::-1]
        tv = orc.verify_tree(rows, np.array([0, n], np.int32), tok, parent, 12)
        k = len(want_path)
        assert tv.accept_len[0] == k - 1
        assert tv.path[0, :k].tolist() == want_path
        assert tv.out_tokens[0, :k - 1].tolist() == [int(tok[j]) for j in want_path[1:]]
        assert tv.out_tokens[0, k - 1] == am[want_path[-1]]


def _anc(parent, j):
    out = [j]
    while parent[j] >= 0:
        j = int(parent[j])
        out.append(j)
    return out


@pytest.mark.parametrize("width", [4, 8, 12, 16])
def test_planted_paths_of_the_tree_workload_are_recovered(orc, width):
    cfg = W.tree_bs32(width=width, B=8)
    tb = orc.build_tree(cfg["anchor"], cfg["cand_tok"], cfg["cand_score"], cfg["ng_tok"], cfg["ng_len"],
                        cfg["ng_score"], cfg["ng_adj"], width)
    node_off, tok, parent = W.flatten_trees(tb.tok, tb.parent, tb.n_rows)
    logits, planted = W.tree_logits(node_off, tok, parent, cfg["V"])
    tv = orc.verify_tree(logits, node_off, tok, parent, cfg["max_nodes"])
    assert tv.status == 0
    for r, path in enumerate(planted):
        assert tv.path[r, :len(path)].tolist() == path
        assert tv.accept_len[r] == len(path) - 1


@pytest.mark.parametrize("width", [8, 12, 16])
def test_tree_workload_realises_mean_accept_length_3(orc, width):
    """The 32-request tree workload plants paths whose accept lengths average 3
    (the configuration's expected accept length), within 0.5."""
    cfg = W.tree_bs32(width=width)
    tb = orc.build_tree(cfg["anchor"], cfg["cand_tok"], cfg["cand_score"], cfg["ng_tok"], cfg["ng_len"],
                        cfg["ng_score"], cfg["ng_adj"], width)
    node_off, tok, parent = W.flatten_trees(tb.tok, tb.parent, tb.n_rows)
    logits, planted = W.tree_logits(node_off, tok, parent, cfg["V"])
    tv = orc.verify_tree(logits, node_off, tok, parent, cfg["max_nodes"])
    assert [len(p) - 1 for p in planted] == tv.accept_len.tolist()
    assert abs(tv.accept_len.mean() - 3.0) <= 0.5, tv.accept_len.mean()


def test_filled_tree_workload_realises_mean_accept_length_3(orc):
    c = W.tree_fill_bs32(width=16)
    fo = orc.ngram_fill(c["hist"], c["hist_len"], c["cand_tok"], c["n_min"], c["copy_cap"], c["max_depth"], c["Lg"])
    tb = orc.build_tree(c["anchor"], c["cand_tok"], c["cand_score"], fo.tok, fo.len, c["ng_score"], c["ng_adj"], 16)
    node_off, tok, parent = W.flatten_trees(tb.tok, tb.parent, tb.n_rows)
    logits, _ = W.tree_logits(node_off, tok, parent, c["V"])
    tv = orc.verify_tree(logits, node_off, tok, parent, 16)
    assert abs(tv.accept_len.mean() - 3.0) <= 0.5, tv.accept_len.mean()


@pytest.mark.parametrize("depth", [1, 2, 3, 4, 6, 9, 20])
def test_capped_geometric_rate_gives_mean_3_or_the_depth(depth):
    a = W._capped_geometric_rate(depth, 3.0)
    assert 0.0 < a <= 1.0
    mean = sum(a ** k for k in range(1, depth + 1))  # E[min(A, d)] = sum_k P(A >= k)
    assert abs(mean - min(3.0, depth)) < 1e-9


def test_invalid_trees_are_flagged(orc):
    rows = np.zeros((3, 5), np.float32)
    tv = orc.verify_tree(rows, np.array([0, 3], np.int32), np.array([0, 1, 2], np.int32),
                         np.array([-1, 0, 2], np.int32), 4)
    assert tv.status & orc.ST_BAD_TREE and tv.accept_len[0] == -1
    tv = orc.verify_tree(rows, np.array([0, 3], np.int32), np.array([0, 1, 2], np.int32),
                         np.array([-1, 0, 1], np.int32), 2)
    assert tv.status & orc.ST_BAD_LENGTH
