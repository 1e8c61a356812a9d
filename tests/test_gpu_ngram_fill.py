"""GPU parity of the n-gram fill of the candidate tree (spec_ngram_fill) and of
the builder fed with chains from the anchor and from every pick, against the
oracle; then the whole filled tree round (fill, build, greedy tree verify).
Exactness: chain tokens, lengths and evidence bit-exact; trees as in
tests/_gpu.assert_tree_equal."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from ._gpu import assert_tree_equal, gpu_build_tree, gpu_ngram_fill, gpu_tree
from .test_oracle_ngram_fill import _text

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return S


def _check(S, hist, hist_len, cand_tok, n_min, copy_cap, max_depth, Lg, status=0):
    ws = S.Workspace(1, 1, 1, 1)
    g = gpu_ngram_fill(S, ws, hist, hist_len, cand_tok, n_min, copy_cap, max_depth, Lg)
    o = O.ngram_fill(hist, hist_len, cand_tok, n_min, copy_cap, max_depth, Lg)
    np.testing.assert_array_equal(g["len"], o.len)
    np.testing.assert_array_equal(g["tok"], o.tok)
    np.testing.assert_array_equal(g["ev"], o.ev)
    assert ws.status() == status and o.status == status
    return o


@pytest.mark.parametrize("n_min", [1, 2, 4])
def test_fill_parity_on_the_tree_workload(S, n_min):
    c = W.tree_fill_bs32()
    o = _check(S, c["hist"], c["hist_len"], c["cand_tok"], n_min, 256, 32, 32)
    assert o.len[:, 0].min() > 0  # every anchor continues the planted repeat


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("n_min,V,repeats,copy_cap", [(1, 12, 0.5, 256), (4, 12, 0.5, 256), (4, 5, 0.0, 256),
                                                      (2, 6, 0.3, 2), (3, 40, 0.7, 8)])
@pytest.mark.parametrize("stride", [700, 699])  # 699: rows not 16-byte aligned, texts staged token by token
def test_fill_parity_random_texts(S, seed, n_min, V, repeats, copy_cap, stride):
    rng = np.random.default_rng(1000 + seed)
    B, P, Kc = 24, 6, 3
    hist = np.full((B, stride), -5, np.int32)
    hist_len = rng.integers(0, stride + 1, B).astype(np.int32)
    hist_len[:3] = [0, 1, 2]
    for r in range(B):
        hist[r, :hist_len[r]] = _text(rng, int(hist_len[r]), V, repeats) if hist_len[r] > 16 else \
            rng.integers(0, V, hist_len[r])
    cand_tok = rng.integers(0, V, (B, P, Kc)).astype(np.int32)
    _check(S, hist, hist_len, cand_tok, n_min, copy_cap, 32, 40)


@pytest.mark.parametrize("max_depth,Lg", [(0, 8), (3, 8), (32, 5), (9, 64)])
def test_fill_depth_and_capacity(S, max_depth, Lg):
    rng = np.random.default_rng(77)
    hist = np.tile(np.arange(1, 9, dtype=np.int32), 40)[None].repeat(3, 0)
    cand_tok = np.tile(np.arange(1, 9, dtype=np.int32)[:, None], (3, 1, 2))[:, :6]
    cand_tok[1] = rng.integers(1, 9, (6, 2))
    _check(S, hist, np.array([320, 319, 100], np.int32), cand_tok, 1, 256, max_depth, Lg)


def test_fill_long_history(S):
    # 32768-token histories with a long planted repeat (copies capped at 256)
    rng = np.random.default_rng(5)
    B, T = 3, 32768
    hist = np.empty((B, T), np.int32)
    for r in range(B):
        h = W.zipf_tokens(rng, T, 151936)
        at = int(rng.integers(0, T // 2))
        h[T - 300:] = h[at:at + 300]
        hist[r] = h
    cand_tok = W.zipf_tokens(rng, B * 8 * 4, 151936).reshape(B, 8, 4).astype(np.int32)
    _check(S, hist, np.full(B, T, np.int32), cand_tok, 4, 256, 32, 32)


def test_fill_flags_a_bad_length(S):
    hist = np.tile(np.arange(6, dtype=np.int32), 4)[None].repeat(2, 0)
    cand_tok = np.zeros((2, 2, 1), np.int32)
    o = _check(S, hist, np.array([24, 25], np.int32), cand_tok, 1, 256, 32, 8, status=S.DEV_BITS["bad_length"])
    assert o.len[1].tolist() == [0, 0, 0]


@pytest.mark.parametrize("n_fol,reps,extra", [(2100, 1, (1700,)), (2049, 1, ()), (5000, 1, (4321, 17)),
                                               (3000, 2, (2999, 5, 2999)), (16000, 1, (9, 15999))])
def test_fill_counts_more_followers_than_the_table_exactly(S, n_fol, reps, extra):
    """"1 2 3" followed by n_fol distinct tokens (each `reps` times), some of
    them once more, then a context whose 4-token suffix is new: more distinct
    followers than the 2048-entry on-chip table holds.  The chains equal the
    oracle's, which counts every follower, and no status bit is set; the
    16,000-follower text (64,004 tokens) is too long to stage on chip."""
    body = np.stack([np.ones(n_fol), 2 * np.ones(n_fol), 3 * np.ones(n_fol), 1000 + np.arange(n_fol)], 1).ravel()
    parts = [body] * reps + [np.array([1, 2, 3, 1000 + k]) for k in extra] + [np.array([99, 1, 2, 3])]
    hist = np.concatenate(parts).astype(np.int32)[None]
    o = _check(S, hist, np.array([hist.shape[1]], np.int32), np.zeros((1, 0, 1), np.int32), 4, 256, 32, 8)
    assert o.len[0, 0] > 0
    want = 1000 + (extra[-1] if extra else n_fol - 1)  # most frequent, then most recent
    assert o.tok[0, 0, 0] == want


# ------------------------------------------------------------------ the builder with chains from every pick
def _random_chain_blocks(seed, B, P, Kc, Lg):
    rng = np.random.default_rng(seed)
    cand_tok = np.stack([np.stack([rng.choice(40, Kc, replace=False) for _ in range(P)]) for _ in range(B)]) \
        if P > 0 else np.zeros((B, 0, Kc), np.int32)
    ng = np.full((B, P + 1, Lg), -1, np.int32)
    ln = np.zeros((B, P + 1), np.int32)
    for r in range(B):
        for c in range(P + 1):
            pos, k = c, 0
            for _ in range(int(rng.integers(0, Lg + 1))):
                if pos < P and rng.random() < 0.6:
                    ng[r, c, k] = cand_tok[r, pos, 0 if rng.random() < 0.7 else int(rng.integers(0, Kc))]
                    pos += 1
                else:
                    ng[r, c, k] = 1000 + int(rng.integers(0, 3))  # few values: chains meet again
                    pos = P
                k += 1
            ln[r, c] = k
    return dict(anchor=rng.integers(0, 40, B).astype(np.int32), cand_tok=cand_tok.astype(np.int32),
                cand_score=rng.normal(0, 1.5, (B, P, Kc)).astype(np.float32), ng_tok=ng, ng_len=ln,
                ng_score=rng.normal(0, 1, B).astype(np.float32), ng_adj=np.abs(rng.normal(0, 1, B)).astype(np.float32))


@pytest.mark.parametrize("P,Kc,Lg,width", [(8, 4, 12, 16), (8, 4, 32, 64), (3, 2, 6, 256), (12, 3, 30, 200),
                                           (1, 1, 5, 4), (0, 2, 9, 8),
                                           # 21 and 32 chains: the parallel merge at its widest (496 chain
                                           # pairs); 41 chains: the depth-by-depth merge
                                           (20, 3, 12, 64), (31, 4, 8, 128), (40, 2, 8, 32)])
def test_builder_parity_with_chains_from_every_pick(S, P, Kc, Lg, width):
    c = _random_chain_blocks(P * 100 + Lg, 40, P, Kc, Lg)
    args = (c["anchor"], c["cand_tok"], c["cand_score"], c["ng_tok"], c["ng_len"], c["ng_score"], c["ng_adj"])
    ws = S.Workspace(40, 1, 1, 1)
    g = gpu_build_tree(S, ws, *args, width)
    o = O.build_tree(*args, width)
    assert_tree_equal(g, o)
    assert ws.status() == 0


@pytest.mark.parametrize("width", [4, 8, 16, 32])
def test_filled_tree_round(S, width):
    c = W.tree_fill_bs32(width=width)
    ws = S.Workspace(c["B"], 1, 1, 1)
    gf = gpu_ngram_fill(S, ws, c["hist"], c["hist_len"], c["cand_tok"], c["n_min"], c["copy_cap"], c["max_depth"],
                        c["Lg"])
    of = O.ngram_fill(c["hist"], c["hist_len"], c["cand_tok"], c["n_min"], c["copy_cap"], c["max_depth"], c["Lg"])
    np.testing.assert_array_equal(gf["tok"], of.tok)
    args = (c["anchor"], c["cand_tok"], c["cand_score"], gf["tok"], gf["len"], c["ng_score"], c["ng_adj"])
    g = gpu_build_tree(S, ws, *args, width)
    o = O.build_tree(*args, width)
    assert_tree_equal(g, o)
    node_off, tok, parent = W.flatten_trees(g["tok"], g["parent"], g["n_rows"])
    logits, planted = W.tree_logits(node_off, tok, parent, c["V"])
    ws2 = S.Workspace(c["B"], int(node_off[-1]), 1, c["V"])
    gv = gpu_tree(S, ws2, logits, node_off, tok, parent, width)
    ov = O.verify_tree(logits, node_off, tok, parent, width)
    assert np.array_equal(gv["path"], ov.path) and np.array_equal(gv["out"], ov.out_tokens)
    assert ws.status() == 0 and ws2.status() == 0
