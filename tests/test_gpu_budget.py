"""GPU parity of budget sizing (spec_size_budget) against the oracle, and the
two-step stale pipeline of round.BudgetSizer.  Exactness: b* equal, except
where the oracle's G has a near-tie (relative gap <= 1e-12) between the two
answers (the kernel sums by segments, the oracle left to right); lambda within
1e-6 relative (one fp32 rounding of nearly equal doubles)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return S


def _gpu(S, Sv, chain_len, mvl, C0, p):
    ws = S.Workspace(1, 1, 1, 1)
    b = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    lam = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    S.spec_size_budget(torch.as_tensor(np.ascontiguousarray(Sv, np.float32)).cuda(),
                       torch.as_tensor(np.ascontiguousarray(chain_len, np.int32)).cuda(), mvl, C0, p, b, lam, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return int(b.item()), float(lam.item())


def _check(S, Sv, chain_len, mvl, C0, p):
    o = O.size_budget(Sv, chain_len, mvl, C0, p)
    b, lam = _gpu(S, Sv, chain_len, mvl, C0, p)
    if b != o.b_star:
        assert abs(o.G[b] - o.G[o.b_star]) <= 1e-12 * o.G[o.b_star], (b, o.b_star)
    assert abs(lam - np.float32(o.lam)) <= 1e-6 * max(abs(o.lam), 1e-30)
    return b, o


def _priced(c):
    ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
    return O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                                c["coef"], c["lam"], c["budget"], c["max_verify_len"], c["policy"],
                                c["draft_greedy"])


@pytest.mark.parametrize("name", ["tiny", "edit_bs4", "mixed_bs128", "long_bs64"])
@pytest.mark.parametrize("C0,p", [(20.0, 1.0), (100.0, 0.5), (5.0, 3.0)])
def test_budget_parity_on_priced_workloads(S, name, C0, p):
    c = {"tiny": W.tiny, "edit_bs4": W.edit_bs4, "mixed_bs128": W.mixed_bs128, "long_bs64": W.long_bs64}[name]()
    pr = _priced(c)
    _check(S, pr.S, pr.chain_len, c["max_verify_len"], C0 * c["B"] / 8, p)


@pytest.mark.parametrize("B,L,seed", [(1, 1, 0), (3, 15, 1), (100, 15, 2), (1024, 31, 3), (257, 7, 4), (128, 16, 5),
                                        (129, 16, 6)])
def test_budget_parity_random(S, B, L, seed):
    rng = np.random.default_rng(seed)
    Sv = np.cumprod(rng.uniform(0.3, 1.0, (B, L)), axis=1).astype(np.float32)
    chain_len = rng.integers(0, L + 1, B).astype(np.int32)
    for C0, p in [(B * 2.0, 1.0), (B * 0.2, 0.05), (10.0, 10.0)]:
        _check(S, Sv, chain_len, int(rng.integers(0, L + 1)), C0, p)


def test_budget_degenerate_cases(S):
    # no batch; no verifiable slot; equal survivals making G constant (the smallest b wins)
    assert _gpu(S, np.zeros((0, 4), np.float32), np.zeros(0, np.int32), 4, 1.0, 1.0) == (0, 0.0)
    b, lam = _gpu(S, np.ones((3, 4), np.float32), np.zeros(3, np.int32), 4, 6.0, 1.0)
    assert b == 0 and lam == np.float32(0.5)
    b, lam = _gpu(S, np.full((4, 5), 0.5, np.float32), np.full(4, 5, np.int32), 5, 8.0, 1.0)
    assert b == 0 and lam == np.float32(0.5)


def test_stale_pipeline_uses_the_survivals_of_two_steps_before(S):
    from speculative_decoding_draft_spec_gb300.round import BudgetSizer, ChainRound

    c = W.mixed_bs128()
    B, K, L, V = c["B"], c["K"], c["L"], c["V"]
    rnd = ChainRound(B, c["hist"].shape[1], K, L, V, torch.bfloat16, 16, c["coef"], c["n_min"], c["n_max"],
                     c["copy_cap"])
    sizer = BudgetSizer(C0=256.0, p=1.0, budget0=c["budget"], lam0=c["lam"], max_verify_len=L)
    lens = np.array(c["hist_len"])
    used, sized_from = [], []
    for step in range(5):
        # a slightly different batch each step: the histories grow by one token
        rnd.load(c["hist"], lens + step, c["d"], c["c"], c["d_len"])
        budget, lam = sizer.params(step)
        used.append((budget, lam))
        sizer.before_next_step()
        rnd.draft_and_price(lam, budget, L, c["policy"], True)
        sizer.size(rnd, step)
        torch.cuda.synchronize()
        sized_from.append((rnd.S.cpu().numpy().copy(), rnd.chain_len.cpu().numpy().copy()))
    assert used[0] == used[1] == (c["budget"], float(c["lam"]))
    for step in range(2, 5):
        o = O.size_budget(*sized_from[step - 2], L, 256.0, 1.0)
        b, lam = used[step]
        if b != o.b_star:
            assert abs(o.G[b] - o.G[o.b_star]) <= 1e-12 * o.G[o.b_star]
        assert abs(lam - np.float32(o.lam)) <= 1e-6 * o.lam


def test_survival_outside_unit_interval_is_flagged_and_clamped(S):
    Sv = np.full((2, 3), 0.6, np.float32)
    Sv[1, 0] = 1.5
    ws = S.Workspace(1, 1, 1, 1)
    b = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    lam = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    S.spec_size_budget(torch.as_tensor(Sv).cuda(), torch.full((2,), 3, dtype=torch.int32, device="cuda"), 3, 4.0, 1.0,
                       b, lam, ws)
    torch.cuda.synchronize()
    assert ws.status() & 0x10
    o = O.size_budget(np.clip(Sv, 0, 1), np.full(2, 3, np.int32), 3, 4.0, 1.0)
    assert int(b.item()) == o.b_star
