"""GPU parity of the candidate-tree builder (spec_build_tree) against the
oracle, and the whole tree round (build, then greedy tree verification) on the
batch-32 tree workload.  Exactness: rows, parents and candidate ids bit-exact,
except among candidates whose Q ties at the selection cut within 1e-12
(tests/_gpu.assert_tree_equal)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from ._gpu import assert_tree_equal, gpu_build_tree, gpu_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return S


def _both(S, c, width, ws=None):
    ws = ws or S.Workspace(len(c["anchor"]), 1, 1, 1)
    args = (c["anchor"], c["cand_tok"], c["cand_score"], c["ng_tok"], c["ng_len"], c["ng_score"], c["ng_adj"])
    g = gpu_build_tree(S, ws, *args, width)
    o = O.build_tree(*args, width)
    return g, o, ws


@pytest.mark.parametrize("width", [1, 2, 4, 8, 12, 16, 64])
def test_tree_build_parity_on_the_tree_workload(S, width):
    c = W.tree_bs32(width=min(width, 16))
    g, o, ws = _both(S, c, width)
    assert_tree_equal(g, o)
    assert ws.status() == 0


def _random_blocks(seed, B, P, Kc, Lg, tie=False):
    rng = np.random.default_rng(seed)
    cand_tok = np.stack([np.stack([rng.choice(60, Kc, replace=False) for _ in range(P)]) for _ in range(B)]) \
        if P > 0 else np.zeros((B, 0, Kc), np.int64)
    score = rng.normal(0, 1.5, (B, P, Kc))
    if tie:
        score = np.round(score)  # many exact ties
    ng = rng.integers(0, 60, (B, max(Lg, 1)))
    for r in range(B):  # some chains follow picks or siblings for a while
        k = int(rng.integers(0, min(P, Lg) + 1))
        for i in range(k):
            ng[r, i] = cand_tok[r, i, 0 if rng.random() < 0.7 else int(rng.integers(0, Kc))]
    return dict(anchor=rng.integers(0, 60, B), cand_tok=cand_tok.astype(np.int32), cand_score=score.astype(np.float32),
                ng_tok=ng.astype(np.int32), ng_len=rng.integers(0, Lg + 1, B).astype(np.int32),
                ng_score=rng.normal(0, 1, B).astype(np.float32), ng_adj=np.abs(rng.normal(0, 1, B)).astype(np.float32))


@pytest.mark.parametrize("P,Kc,Lg,width,tie", [
    (8, 4, 15, 16, False), (8, 4, 15, 33, True), (0, 3, 20, 8, False), (6, 1, 0, 5, False),
    (16, 8, 32, 161, False), (31, 8, 7, 256, True), (2, 3, 3, 3, True), (1, 1, 1, 256, False)])
def test_tree_build_parity_random_blocks(S, P, Kc, Lg, width, tie):
    c = _random_blocks(P * 1000 + Kc * 10 + Lg, 40, P, Kc, Lg, tie)
    g, o, ws = _both(S, c, width)
    assert_tree_equal(g, o)
    assert ws.status() == 0


def test_tree_build_deep_spine(S):
    # one pick per position: a spine 200 deep, then a 55-token chain below it
    P, Kc, Lg = 200, 1, 55
    rng = np.random.default_rng(9)
    c = dict(anchor=np.array([1, 2], np.int32), cand_tok=rng.integers(0, 9, (2, P, Kc)).astype(np.int32),
             cand_score=rng.normal(3, 0.5, (2, P, Kc)).astype(np.float32), ng_len=np.array([Lg, 3], np.int32),
             ng_score=np.array([2.0, 0.0], np.float32), ng_adj=np.array([0.5, 0.0], np.float32))
    ng = rng.integers(100, 200, (2, Lg)).astype(np.int32)
    ng[0, :P // 4] = c["cand_tok"][0, :P // 4, 0]
    c["ng_tok"] = ng
    g, o, ws = _both(S, c, 256)
    assert_tree_equal(g, o)


def test_tree_build_flags_bad_chain_lengths(S):
    c = _random_blocks(5, 4, 3, 2, 4)
    c["ng_len"] = np.array([2, -1, 5, 4], np.int32)  # -1 and 5 lie outside [0, Lg]
    g, o, ws = _both(S, c, 8)
    assert o.status & O.ST_BAD_LENGTH and ws.status() & S.DEV_BITS["bad_length"]
    assert_tree_equal(g, o)


@pytest.mark.parametrize("width", [4, 8, 12, 16])
def test_tree_round_build_then_verify(S, width):
    c = W.tree_bs32(width=width)
    g, o, ws = _both(S, c, width)
    assert_tree_equal(g, o)
    node_off, tok, parent = W.flatten_trees(g["tok"], g["parent"], g["n_rows"])
    logits, planted = W.tree_logits(node_off, tok, parent, c["V"])
    ws2 = S.Workspace(c["B"], int(node_off[-1]), 1, c["V"])
    gv = gpu_tree(S, ws2, logits, node_off, tok, parent, width)
    ov = O.verify_tree(logits, node_off, tok, parent, width)
    assert np.array_equal(gv["path"], ov.path) and np.array_equal(gv["accept_len"], ov.accept_len)
    assert np.array_equal(gv["out"], ov.out_tokens)
    for r, p in enumerate(planted):
        assert gv["path"][r, :len(p)].tolist() == p
    assert ws2.status() == 0
