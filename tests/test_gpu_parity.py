"""GPU parity: every step through the C ABI against the oracle on the same
seeded inputs, at the workloads' full sizes and at small sizes that still
span several units and a ragged tail, plus the edge cases.

Exactness: token ids, proposals, features, budget selections, survivals,
greedy accept lengths and tree paths bit-exact; sampled decisions per
tests/_gpu.compare_sampled (|u - ratio| < 1e-5 band, residual within 1e-5)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from ._gpu import (compare_sampled, gpu_chain, gpu_draft_price, gpu_ngram, gpu_price, gpu_tree, host,
                   logits_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return S


def _ws(S, B, rows, K, V):
    return S.Workspace(B, max(rows, 1), K, V)


# ------------------------------------------------------------------ estimator
COEFS = [("table5_qwen3_4b", W.table5_coef()), ("table5_n_full_4", W.table5_coef(n_full=4)),
         ("table5_llama", W.table5_coef("llama3_1_8b"))] + \
        [(f"table7_{i}", W.table7_coef(i)) for i in range(1, 6)] + [("constant", W.constant_coef(0.9))]


@pytest.mark.parametrize("name,coef", COEFS, ids=[c[0] for c in COEFS])
def test_estimator_table_equals_oracle_on_every_key(S, name, coef):
    L = 15
    est = S.EstimatorTable(coef, L)
    tab = host(est.table)
    if coef.get("constant_h") is not None:
        assert tab[0] == O.estimate_h(coef, 1, 5, 1, 5)
        return
    mcap = coef["m_cap"]
    nf = coef["n_full"]
    mism = []
    for k in range(1, L + 1):
        for n in range(0, 33):
            if n == nf:
                continue
            for a in (0, 1):
                got = tab[(n * 2 + a) * L + (k - 1)]
                if got != O.estimate_h(coef, k, n, a, n):
                    mism.append((k, n, a))
        for a in (0, 1):
            for m in range(1, mcap + 1):
                if tab[L * 66 + (a * (mcap + 1) + m) * L + (k - 1)] != O.estimate_h(coef, k, nf, a, m):
                    mism.append((k, nf, a, m))
    assert not mism, mism[:10]


# ------------------------------------------------------------------ n-gram
def _cfg_hist(name):
    if name == "tiny":
        c = W.tiny()
    elif name == "edit_bs4":
        c = W.edit_bs4()
    elif name == "mixed_bs128":
        c = W.mixed_bs128()
    elif name == "long_bs64":
        c = W.long_bs64()
    else:
        t = W.tree_bs32(width=4, B=32)
        return t["hist"], np.full(32, 4096, np.int32), 5, 15
    return c["hist"], c["hist_len"], c["n_min"], c["n_max"]


@pytest.mark.parametrize("name", ["tiny", "edit_bs4", "mixed_bs128", "long_bs64", "tree_hist"])
def test_ngram_parity_on_workloads(S, name):
    hist, hist_len, n_min, n_max = _cfg_hist(name)
    ws = _ws(S, hist.shape[0], 1, 1, 1)
    g = gpu_ngram(S, ws, hist, hist_len, n_min, n_max)
    o = O.ngram_propose(hist, hist_len, n_min, n_max, 15, 256)
    for got, want in zip(g, (o.g, o.g_len, o.match_n, o.agree, o.copy_len)):
        assert np.array_equal(got, want)
    assert ws.status() == 0
    assert (o.g_len > 0).any()


@pytest.mark.parametrize("stride", [64, 67, 256, 1000])
def test_ngram_parity_small_alphabets_and_edges(S, stride):
    rng = np.random.default_rng(stride)
    B = 48
    hist = rng.integers(0, 3, (B, stride)).astype(np.int32)
    hist[:8] = np.tile([4, 5, 6, 7], stride // 4 + 1)[:stride]  # periodic
    hist_len = rng.integers(0, stride + 1, B).astype(np.int32)
    hist_len[:6] = [0, 1, 2, 3, stride, stride - 1]
    ws = _ws(S, B, 1, 1, 1)
    for n_min, n_max, cap in [(1, 3, 256), (2, 5, 5), (5, 15, 256), (1, 1, 1), (3, 32, 40)]:
        g = gpu_ngram(S, ws, hist, hist_len, n_min, n_max, 15, cap)
        o = O.ngram_propose(hist, hist_len, n_min, n_max, 15, cap)
        for got, want in zip(g, (o.g, o.g_len, o.match_n, o.agree, o.copy_len)):
            assert np.array_equal(got, want), (n_min, n_max, cap)


def test_ngram_bad_lengths_are_flagged(S):
    hist = np.arange(64, dtype=np.int32).reshape(2, 32) % 5
    ws = _ws(S, 2, 1, 1, 1)
    g = gpu_ngram(S, ws, hist, np.array([33, -1], np.int32), 1, 3)
    assert ws.status() & S.DEV_BITS["bad_length"]
    assert np.all(g[1] == 0) and np.all(g[0] == -1)


# ------------------------------------------------------------------ pricing
def _priced_inputs(c):
    o = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
    return o


def _price_both(S, c, ng, policy=None, greedy=None, budget=None, lam=None, mvl=None):
    B, K = c["d"].shape
    policy = c["policy"] if policy is None else policy
    greedy = c["draft_greedy"] if greedy is None else greedy
    budget = c["budget"] if budget is None else budget
    lam = c["lam"] if lam is None else lam
    mvl = c["max_verify_len"] if mvl is None else mvl
    est = S.EstimatorTable(c["coef"], c["L"])
    ws = _ws(S, B, 1, K, 1)
    g = gpu_price(S, ws, est, c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                  lam, budget, mvl, policy, greedy)
    o = O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                             c["coef"], lam, budget, mvl, policy, greedy)
    return g, o, ws


def _assert_price_equal(g, o):
    for k in ("chain", "chain_len", "source", "verify_len", "row_off", "point_mass"):
        assert np.array_equal(g[k], getattr(o, k)), k
    assert np.array_equal(g["S"].view(np.uint32), o.S.view(np.uint32))  # bit for bit


@pytest.mark.parametrize("name", ["tiny", "tiny_prob", "edit_bs4", "edit_bs4_prob", "mixed_bs128", "long_bs64"])
def test_price_parity_on_workloads(S, name):
    c = {"tiny": lambda: W.tiny(), "tiny_prob": lambda: W.tiny(probabilistic=True),
         "edit_bs4": lambda: W.edit_bs4(), "edit_bs4_prob": lambda: W.edit_bs4(temperature=1.0, probabilistic=True),
         "mixed_bs128": W.mixed_bs128, "long_bs64": W.long_bs64}[name]()
    ng = _priced_inputs(c)
    g, o, ws = _price_both(S, c, ng)
    _assert_price_equal(g, o)
    assert ws.status() == 0
    assert o.verify_len.sum() == min(c["budget"], int(np.minimum(o.chain_len, c["max_verify_len"]).sum()))


def test_price_parity_random_stress(S):
    rng = np.random.default_rng(31)
    for trial in range(40):
        B = int(rng.integers(1, 300))
        K, L = 7, 15
        d = rng.integers(0, 20, (B, K)).astype(np.int32)
        g = np.full((B, L), -1, np.int32)
        g_len = rng.integers(0, L + 1, B).astype(np.int32)
        for r in range(B):
            g[r, :g_len[r]] = rng.integers(0, 20, g_len[r])
            if rng.random() < 0.3 and g_len[r] > K:  # contains d
                g[r, :K] = d[r]
        cvals = rng.choice([0.5, 0.9, 0.95, 1.0, rng.random()], (B, K)).astype(np.float32)
        n = rng.integers(0, 17, B).astype(np.int32)
        n[rng.random(B) < 0.3] = 15
        a = rng.integers(0, 2, B).astype(np.int32)
        m = np.maximum(n, rng.integers(0, 400, B)).astype(np.int32)
        cfg = dict(d=d, c=cvals, d_len=rng.integers(0, K + 1, B).astype(np.int32), L=L,
                   coef=[W.table5_coef(), W.table7_coef(1), W.constant_coef(0.9)][trial % 3])
        ng = O.NgramOut(g, g_len, n, a, m, 0)
        budget = int(rng.integers(0, B * L + 5))
        policy = ["proposed", "ngram_first", "extension", "model_only", "ngram_only"][trial % 5]
        gp, op, ws = _price_both(S, cfg, ng, policy=policy, greedy=bool(trial % 2), budget=budget,
                                 lam=float(rng.choice([0.0, 0.04, 0.3, 0.9])), mvl=int(rng.integers(0, 17)))
        _assert_price_equal(gp, op)


@pytest.mark.parametrize("kind", ["copies", "distinct", "copies_and_distinct"])
@pytest.mark.parametrize("B", [128, 300])
def test_price_crowded_value_bin(S, kind, B):
    """More than 256 keys within one 1/1024 of survival value, where the budget's
    threshold falls: copies of one key (confidences of exactly 1), distinct
    keys (confidences just below 1), or both.  Batch 300 keeps the keys in
    shared memory only, batch 128 also in registers."""
    rng = np.random.default_rng(B + len(kind))
    K, L = 7, 15
    if kind == "copies":
        c = np.ones((B, K), np.float32)
    elif kind == "distinct":
        c = (1.0 - rng.random((B, K)) * 1e-4).astype(np.float32)
    else:
        c = np.where(rng.random((B, K)) < 0.5, 1.0, 1.0 - rng.random((B, K)) * 1e-4).astype(np.float32)
    cfg = dict(d=rng.integers(0, 50, (B, K)).astype(np.int32), c=c, d_len=np.full(B, K, np.int32), L=L,
               coef=W.table5_coef())
    ng = O.NgramOut(np.full((B, L), -1, np.int32), np.zeros(B, np.int32), np.zeros(B, np.int32),
                    np.zeros(B, np.int32), np.zeros(B, np.int32), 0)
    for budget in (1, 257, B * K // 2 + 1, B * K - 1):
        g, o, ws = _price_both(S, cfg, ng, policy="model_only", greedy=True, budget=budget, lam=0.04, mvl=15)
        _assert_price_equal(g, o)
        assert int(o.verify_len.sum()) == budget
        assert ws.status() == 0


def test_price_flags_out_of_range_confidences(S):
    cfg = dict(d=np.zeros((2, 7), np.int32), c=np.array([[1.5] * 7, [-0.2] * 7], np.float32),
               d_len=np.full(2, 7, np.int32), L=15, coef=W.table5_coef())
    ng = O.NgramOut(np.full((2, 15), -1, np.int32), np.zeros(2, np.int32), np.zeros(2, np.int32),
                    np.zeros(2, np.int32), np.zeros(2, np.int32), 0)
    g, o, ws = _price_both(S, cfg, ng, policy="model_only", greedy=True, budget=5, lam=0.1, mvl=15)
    _assert_price_equal(g, o)
    assert ws.status() & S.DEV_BITS["bad_value"]


# ------------------------------------------------------------------ fused steps 1 + 2
def _fused_vs_oracle(S, c, policy=None, greedy=None, budget=None, lam=None, mvl=None):
    policy = c["policy"] if policy is None else policy
    greedy = c["draft_greedy"] if greedy is None else greedy
    budget = c["budget"] if budget is None else budget
    lam = c["lam"] if lam is None else lam
    mvl = c["max_verify_len"] if mvl is None else mvl
    B, K = c["d"].shape
    est = S.EstimatorTable(c["coef"], c["L"])
    ws = _ws(S, B, 1, K, 1)
    got = gpu_draft_price(S, ws, est, c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["copy_cap"], c["d"],
                          c["c"], c["d_len"], lam, budget, mvl, policy, greedy, L=c["L"])
    ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
    for k, want in (("g", ng.g), ("g_len", ng.g_len), ("match_n", ng.match_n), ("agree", ng.agree),
                    ("copy_len", ng.copy_len)):
        assert np.array_equal(got[k], want), k
    o = O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                             c["coef"], lam, budget, mvl, policy, greedy)
    _assert_price_equal(got, o)
    return got, o, ws


@pytest.mark.parametrize("name", ["tiny", "tiny_prob", "edit_bs4", "edit_bs4_prob", "mixed_bs128", "long_bs64"])
def test_fused_draft_and_price_on_workloads(S, name):
    c = {"tiny": lambda: W.tiny(), "tiny_prob": lambda: W.tiny(probabilistic=True),
         "edit_bs4": lambda: W.edit_bs4(), "edit_bs4_prob": lambda: W.edit_bs4(temperature=1.0, probabilistic=True),
         "mixed_bs128": W.mixed_bs128, "long_bs64": W.long_bs64}[name]()
    got, o, ws = _fused_vs_oracle(S, c)
    assert ws.status() == 0
    # called twice in a row: the arrival counter is back at zero
    got2, _, _ = _fused_vs_oracle(S, c)
    assert np.array_equal(got2["row_off"], o.row_off)


@pytest.mark.parametrize("L", [15, 31])
@pytest.mark.parametrize("B", [1, 9, 10, 11, 32, 33])
def test_fused_draft_and_price_small_batch_paths(S, B, L):
    """Batches around the bounds of the small-batch allocation paths: request
    counts carried in the arrival (at most 10 requests), the one-warp path (at
    most 32), the block-wide selection; budgets of zero, of every valid slot,
    and of part of them; chains of up to 15 and of up to 31 slots (a request's
    count field must hold 31).  Each call twice in a row (the arrival words
    return to zero)."""
    rng = np.random.default_rng(700 + B + L)
    K, stride = 7, 300
    hist = rng.integers(0, 5, (B, stride)).astype(np.int32)
    hist_len = rng.integers(2, stride + 1, B).astype(np.int32)
    d = np.where(rng.random((B, K)) < 0.5, hist[:, :K], rng.integers(0, 5, (B, K))).astype(np.int32)
    c = {"hist": hist, "hist_len": hist_len, "n_min": 1, "n_max": 4, "copy_cap": 256, "d": d,
         "c": rng.choice([0.5, 0.9, 1.0, 0.3], (B, K)).astype(np.float32),
         "d_len": rng.integers(0, K + 1, B).astype(np.int32), "L": L, "coef": W.table5_coef(n_full=4)}
    for budget in (0, B * L, max(1, B * L // 3)):
        for _ in range(2):
            got, o, ws = _fused_vs_oracle(S, c, policy="proposed", greedy=True, budget=budget, lam=0.04, mvl=L)
            assert ws.status() == 0
    if L == 31:  # some request's chain fills all 31 slots
        assert int(o.chain_len.max()) == 31


def test_fused_draft_and_price_random_stress(S):
    rng = np.random.default_rng(41)
    for trial in range(30):
        B = int(rng.integers(1, 200))
        stride = int(rng.choice([37, 64, 300, 2048]))
        K, L = 7, 15
        hist = rng.integers(0, int(rng.choice([2, 3, 5, 50])), (B, stride)).astype(np.int32)
        hist_len = rng.integers(0, stride + 1, B).astype(np.int32)
        d = np.where(rng.random((B, K)) < 0.5, hist[:, :K], rng.integers(0, 5, (B, K))).astype(np.int32)
        c = {"hist": hist, "hist_len": hist_len, "n_min": int(rng.integers(1, 4)), "copy_cap": 256,
             "d": d, "c": rng.choice([0.5, 0.9, 1.0, 0.3], (B, K)).astype(np.float32),
             "d_len": rng.integers(0, K + 1, B).astype(np.int32), "L": L,
             "coef": [W.table5_coef(n_full=6), W.table7_coef(3), W.constant_coef(0.9)][trial % 3]}
        c["n_max"] = int(rng.integers(c["n_min"], 7))
        _fused_vs_oracle(S, c, policy=["proposed", "ngram_first", "extension", "model_only", "ngram_only"][trial % 5],
                         greedy=bool(trial % 2), budget=int(rng.integers(0, B * L + 3)),
                         lam=float(rng.choice([0.0, 0.04, 0.3])), mvl=int(rng.integers(0, 16)))


# ------------------------------------------------------------------ chain verification
def _layout(S, c, ng=None):
    ng = ng or _priced_inputs(c)
    o = O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                             c["coef"], c["lam"], c["budget"], c["max_verify_len"], c["policy"],
                             c["draft_greedy"])
    return o


@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("prob", [False, True])
def test_chain_tiny_materialised_rows(S, T, prob):
    c = W.tiny(probabilistic=prob, temperature=max(T, 1.0))
    lay = _layout(S, c)
    ro = c["row_off_materialised"]
    draft = c["draft_logits"] if prob else None
    ws = _ws(S, c["B"], int(ro[-1]), c["K"], c["V"])
    for step in range(25 if T > 0 else 1):
        g = gpu_chain(S, ws, c["target_logits"], ro, lay.chain, lay.verify_len, lay.point_mass, draft, T,
                      seed=c["seed"], step=step)
        o = O.verify_chain(c["target_logits"], ro, lay.chain, lay.verify_len, lay.point_mass, draft, T,
                           c["seed"], step)
        if T == 0:
            assert np.array_equal(g["out"], o.out_tokens) and np.array_equal(g["na"], o.n_accepted)
            assert np.array_equal(g["ne"], o.n_emitted)
        else:
            compare_sampled(g, o, c["target_logits"], ro, lay.chain, lay.verify_len, lay.point_mass, draft, T)
    assert ws.status() == 0


def _chain_edit_vs_oracle(S, c, T):
    lay = _layout(S, c)
    logits = W.compact_logits(c, lay.row_off, lay.verify_len)
    draft = c["draft_logits"]
    ws = _ws(S, c["B"], int(lay.row_off[-1]), c["K"], c["V"])
    lt = logits_dev(logits)
    dt = None if draft is None else logits_dev(draft)
    for step in range(8 if T > 0 else 1):
        g = gpu_chain(S, ws, None, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, draft, T,
                      seed=0, step=step, logits_t=lt, draft_t=dt)
        o = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, draft, T, 0, step)
        if T == 0:
            assert np.array_equal(g["out"], o.out_tokens) and np.array_equal(g["na"], o.n_accepted)
            assert np.array_equal(g["ne"], o.n_emitted)
        else:
            compare_sampled(g, o, logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, draft, T)
    assert ws.status() == 0
    return lay


@pytest.mark.parametrize("T,prob", [(0.0, False), (1.0, False), (1.0, True)])
def test_chain_edit_bs4_full_vocab(S, T, prob):
    _chain_edit_vs_oracle(S, W.edit_bs4(temperature=T, probabilistic=prob), T)


# the code-editing configuration swept over its edit rates, all four requests at one rate
EDIT_RATES = [0.0, 0.15, 0.30, 0.45, 0.60, 0.70]


@pytest.mark.parametrize("rate", EDIT_RATES)
@pytest.mark.parametrize("T,prob", [(0.0, False), (1.0, False), (1.0, True)])
def test_chain_edit_bs4_by_edit_rate(S, rate, T, prob):
    _chain_edit_vs_oracle(S, W.edit_bs4(temperature=T, probabilistic=prob, edit_rates=[rate] * 4), T)


@pytest.mark.parametrize("rate", EDIT_RATES)
@pytest.mark.parametrize("prob", [False, True])
def test_fused_draft_and_price_by_edit_rate(S, rate, prob):
    c = W.edit_bs4(temperature=1.0 if prob else 0.0, probabilistic=prob, edit_rates=[rate] * 4)
    got, o, ws = _fused_vs_oracle(S, c)
    assert ws.status() == 0


def test_chain_mixed_bs128_full(S):
    c = W.mixed_bs128()
    lay = _layout(S, c)
    logits = W.compact_logits(c, lay.row_off, lay.verify_len)
    ws = _ws(S, c["B"], int(lay.row_off[-1]), c["K"], c["V"])
    g = gpu_chain(S, ws, logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass)
    o = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass)
    assert np.array_equal(g["out"], o.out_tokens) and np.array_equal(g["na"], o.n_accepted)
    assert np.array_equal(g["ne"], o.n_emitted)
    assert ws.status() == 0
    assert o.n_accepted.sum() > 0


def test_chain_long_bs64_full_fp32_T07(S):
    c = W.long_bs64()
    lay = _layout(S, c)
    ro = c["row_off_materialised"]
    logits = W.materialised_logits(c)
    ws = _ws(S, c["B"], int(ro[-1]), c["K"], c["V"])
    lt = logits_dev(logits)
    for step in range(4):  # four draw sets: accept tests, bonus and correction draws at full size
        g = gpu_chain(S, ws, None, ro, lay.chain, lay.verify_len, lay.point_mass, None, 0.7, step=step,
                      logits_t=lt)
        o = O.verify_chain(logits, ro, lay.chain, lay.verify_len, lay.point_mass, None, 0.7, 0, step)
        st = compare_sampled(g, o, logits, ro, lay.chain, lay.verify_len, lay.point_mass, None, 0.7)
        assert st["exact"] + st["band"] == c["B"]
    assert ws.status() == 0


@pytest.mark.parametrize("V,dtype", [(1000, "bf16"), (2049, "f32"), (4099, "bf16"), (2048, "f32"), (8, "bf16")])
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_chain_ragged_vocab_and_lengths(S, V, dtype, T):
    rng = np.random.default_rng(V)
    B, L, K = 9, 15, 5
    ell = rng.integers(0, L + 1, B).astype(np.int32)
    ell[:2] = [0, L]
    ro = np.concatenate([[0], np.cumsum(ell + 1 + rng.integers(0, 2, B))]).astype(np.int32)  # gaps allowed
    z = (rng.standard_normal((int(ro[-1]), V)) * 2).astype(np.float32)
    chain = rng.integers(0, V, (B, L)).astype(np.int32)
    for r in range(B):  # some leading drafts right
        k = int(rng.integers(0, ell[r] + 1))
        chain[r, :k] = z[ro[r]:ro[r] + k].argmax(1)
    pm = (rng.random((B, L)) < 0.5).astype(np.uint8)
    pm[:, K:] = 1
    draft = (rng.standard_normal((B, K, V)) * 2).astype(np.float32)
    if dtype == "bf16":
        z, draft = W.bf16_bits(z), W.bf16_bits(draft)
    ws = _ws(S, B, int(ro[-1]), K, V)
    for step in range(6 if T > 0 else 1):
        g = gpu_chain(S, ws, z, ro, chain, ell, pm, draft, T, seed=3, step=step)
        o = O.verify_chain(z, ro, chain, ell, pm, draft, T, 3, step)
        if T == 0:
            assert np.array_equal(g["out"], o.out_tokens) and np.array_equal(g["na"], o.n_accepted)
        else:
            compare_sampled(g, o, z, ro, chain, ell, pm, draft, T)
    assert ws.status() == 0


def test_chain_invalid_inputs_are_flagged_not_faulted(S):
    V, B, L = 64, 4, 7
    rng = np.random.default_rng(5)
    z = rng.standard_normal((20, V)).astype(np.float32)
    chain = rng.integers(0, V, (B, L)).astype(np.int32)
    chain[1, 0] = V + 5  # bad token
    ell = np.array([3, 2, 9, 1], np.int32)  # request 2: verify_len > L
    ro = np.array([0, 4, 7, 17, 19], np.int32)  # request 3: rows 17..18 fine
    z[18, 3] = np.nan
    ws = _ws(S, B, 20, 0, V)
    g = gpu_chain(S, ws, z, ro, chain, ell)
    o = O.verify_chain(z, ro, chain, ell)
    st = ws.status()
    assert st & S.DEV_BITS["bad_length"] and st & S.DEV_BITS["bad_token"] and st & S.DEV_BITS["nonfinite"]
    assert o.status & O.ST_BAD_LENGTH and o.status & O.ST_BAD_TOKEN and o.status & O.ST_NONFINITE
    assert np.array_equal(g["out"], o.out_tokens) and np.array_equal(g["na"], o.n_accepted)
    assert np.array_equal(g["ne"], o.n_emitted)
    assert g["ne"][2] == 0 and np.all(g["out"][2] == -1)


# ------------------------------------------------------------------ tree verification
@pytest.mark.parametrize("width", [4, 8, 12, 16])
def test_tree_parity_full_size(S, width):
    t = W.tree_bs32(width=width)
    tb = O.build_tree(t["anchor"], t["cand_tok"], t["cand_score"], t["ng_tok"], t["ng_len"], t["ng_score"],
                      t["ng_adj"], width)
    node_off, tok, parent = W.flatten_trees(tb.tok, tb.parent, tb.n_rows)
    logits, planted = W.tree_logits(node_off, tok, parent, t["V"])
    ws = _ws(S, 32, int(node_off[-1]), 1, t["V"])
    g = gpu_tree(S, ws, logits, node_off, tok, parent, t["max_nodes"])
    o = O.verify_tree(logits, node_off, tok, parent, t["max_nodes"])
    assert np.array_equal(g["path"], o.path) and np.array_equal(g["accept_len"], o.accept_len)
    assert np.array_equal(g["out"], o.out_tokens)
    for r, p in enumerate(planted):
        assert g["path"][r, :len(p)].tolist() == p
    assert ws.status() == 0


def test_tree_random_small_vocab_with_duplicates_and_bad_trees(S):
    rng = np.random.default_rng(77)
    V, B, maxn = 7, 64, 40
    toks, pars, offs = [], [], [0]
    for r in range(B):
        n = int(rng.integers(1, maxn + 1))
        par = np.array([-1] + [int(rng.integers(0, j)) for j in range(1, n)], np.int32)
        tok = rng.integers(0, V, n).astype(np.int32)
        if r % 11 == 5:
            par[n - 1] = n + 3 if n > 1 else 0  # malformed
        toks.append(tok)
        pars.append(par)
        offs.append(offs[-1] + n)
    node_off = np.array(offs, np.int32)
    tok, parent = np.concatenate(toks), np.concatenate(pars)
    z = rng.standard_normal((offs[-1], V)).astype(np.float32)
    for j in range(offs[-1]):  # bias rows toward children's tokens
        z[j, rng.integers(0, V)] += 1.5
    for dt in ("f32", "bf16"):
        zz = z if dt == "f32" else W.bf16_bits(z)
        ws = _ws(S, B, offs[-1], 1, V)
        g = gpu_tree(S, ws, zz, node_off, tok, parent, maxn)
        o = O.verify_tree(zz, node_off, tok, parent, maxn)
        assert np.array_equal(g["path"], o.path) and np.array_equal(g["accept_len"], o.accept_len)
        assert np.array_equal(g["out"], o.out_tokens)
        assert bool(ws.status() & S.DEV_BITS["bad_tree"]) == bool(o.status & O.ST_BAD_TREE)


def test_tree_on_a_chain_equals_greedy_chain_verify_bit_for_bit(S):
    c = W.edit_bs4()
    lay = _layout(S, c)
    logits = W.compact_logits(c, lay.row_off, lay.verify_len)
    ws = _ws(S, c["B"], int(lay.row_off[-1]), c["K"], c["V"])
    gc = gpu_chain(S, ws, logits, lay.row_off, lay.chain, lay.verify_len)
    tok, par = [], []
    for r in range(c["B"]):
        ell = int(lay.verify_len[r])
        tok += [0] + lay.chain[r, :ell].tolist()
        par += list(range(-1, ell))
    gt = gpu_tree(S, ws, logits, lay.row_off, np.array(tok, np.int32), np.array(par, np.int32), 16)
    for r in range(c["B"]):
        n = int(gc["ne"][r])
        assert gt["accept_len"][r] == gc["na"][r]
        assert gt["out"][r, :n].tolist() == gc["out"][r, :n].tolist()


# ------------------------------------------------------------------ the whole round on the device
def test_round_mixed_bs128_on_device_matches_oracle_pipeline(S):
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    c = W.mixed_bs128()
    lay = _layout(S, c)
    logits = W.compact_logits(c, lay.row_off, lay.verify_len)
    rnd = ChainRound(c["B"], c["hist"].shape[1], c["K"], c["L"], c["V"], torch.bfloat16, logits.shape[0],
                     c["coef"], c["n_min"], c["n_max"])
    rnd.load(c["hist"], c["hist_len"], c["d"], c["c"], c["d_len"])
    rnd.logits.copy_(logits_dev(logits))
    rnd.run(c["lam"], c["budget"], c["max_verify_len"])
    torch.cuda.synchronize()
    o = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass)
    assert np.array_equal(host(rnd.row_off), lay.row_off)
    assert np.array_equal(host(rnd.out_tokens), o.out_tokens)
    assert np.array_equal(host(rnd.n_accepted), o.n_accepted)
    # the graph-captured round gives the same result
    rnd.out_tokens.fill_(-9)
    rnd.capture(lam=c["lam"], budget=c["budget"], max_verify_len=c["max_verify_len"])
    rnd.graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(rnd.out_tokens), o.out_tokens)
    assert rnd.ws.status() == 0
