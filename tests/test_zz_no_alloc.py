"""spec_price_and_allocate_static -- pricing with its scratch in the library's
fixed device array instead of a caller workspace -- against
spec_price_and_allocate on the same inputs.

Its outputs must equal the workspace call's bit for bit (the two run the same
kernel), on two calls in a row: the second call only gets them right if the
first left the fixed array's arrival counter at zero.  The largest batch and
chain the array holds (256 requests of 31 slots) are exercised on the device,
and neither torch's allocator nor the device's free memory moves across
calls.  This file is collected last and passes alone or after the other
tests."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    return S


def test_static_pricing_rejects_batches_beyond_its_scratch_without_a_gpu(S):
    lib = S.load()
    e = S.make_estimator({"beta": [0.0] * 15})
    P = 4096  # fake pointer: these calls return before any device work
    INV, UNS = 1, 3

    def price(B, K=7, L=15):
        return lib.spec_price_and_allocate_static(B, K, L, P, P, P, P, P, P, P, P, C.byref(e), P, 1 << 20, 0.1, 8,
                                                  15, 0, 1, P, P, P, P, P, P, P, None, None)

    assert price(257) == UNS  # beyond SPEC_STATIC_PRICE_MAX_BATCH = 256
    assert price(1 << 20) == UNS
    assert price(256, L=40) == UNS
    assert price(256, K=16) == INV
    assert price(-1) == INV


def _inputs(c):
    ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
    return [c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len]


def _run(S, static, est, arrays, lam, budget, mvl, policy, greedy, ws=None, status=None):
    d, c, d_len, g, g_len, n, a, m = [torch.as_tensor(np.ascontiguousarray(x)).cuda() for x in arrays]
    B, L = g.shape
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(chain=torch.full((B, L), -7, **i32), S=torch.full((B, L), -7.0, device="cuda"),
               chain_len=torch.full((B,), -7, **i32), source=torch.full((B,), -7, **i32),
               verify_len=torch.full((B,), -7, **i32), row_off=torch.full((B + 1,), -7, **i32),
               point_mass=torch.full((B, L), 7, dtype=torch.uint8, device="cuda"))
    args = (d, c, d_len, g, g_len, n, a, m, est, lam, budget, mvl, policy, greedy, out["chain"], out["S"],
            out["chain_len"], out["source"], out["verify_len"], out["row_off"], out["point_mass"])
    if static:
        S.spec_price_and_allocate_static(*args, status_word=status)
    else:
        S.spec_price_and_allocate(*args, ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _equal(x, y):
    for k in ("chain", "chain_len", "source", "verify_len", "row_off", "point_mass"):
        assert np.array_equal(x[k], y[k]), k
    assert np.array_equal(x["S"].view(np.uint32), y["S"].view(np.uint32))


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "edit_bs4", "mixed_bs128"])
def test_static_pricing_equals_the_workspace_call_twice_in_a_row(S, name):
    c = {"tiny": W.tiny, "edit_bs4": W.edit_bs4, "mixed_bs128": W.mixed_bs128}[name]()
    arrays = _inputs(c)
    B, K = c["d"].shape
    est = S.EstimatorTable(c["coef"], c["L"])
    ws = S.Workspace(B, 1, K, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    common = (c["lam"], c["budget"], c["max_verify_len"], c["policy"], c["draft_greedy"])
    ref = _run(S, False, est, arrays, *common, ws=ws)
    for _ in range(2):
        _equal(_run(S, True, est, arrays, *common, status=status), ref)
    # two more calls in a row with other budgets, each against its own reference
    for budget in (1, B * c["L"]):
        common = (c["lam"], budget, c["max_verify_len"], c["policy"], c["draft_greedy"])
        _equal(_run(S, True, est, arrays, *common), _run(S, False, est, arrays, *common, ws=ws))
    assert int(status.item()) == 0 and ws.status() == 0


@pytest.mark.gpu
def test_static_pricing_reports_device_errors_in_the_callers_word(S):
    d = np.zeros((2, 7), np.int32)
    conf = np.array([[1.5] * 7, [-0.2] * 7], np.float32)
    arrays = [d, conf, np.full(2, 7, np.int32), np.full((2, 15), -1, np.int32)] + [np.zeros(2, np.int32)] * 4
    est = S.EstimatorTable(W.table5_coef(), 15)
    ws = S.Workspace(2, 1, 7, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    common = (0.1, 5, 15, "model_only", True)
    _equal(_run(S, True, est, arrays, *common, status=status), _run(S, False, est, arrays, *common, ws=ws))
    assert int(status.item()) & S.DEV_BITS["bad_value"]


def _random_inputs(rng, B, K, L):
    d = rng.integers(0, 20, (B, K)).astype(np.int32)
    g = np.full((B, L), -1, np.int32)
    g_len = rng.integers(0, L + 1, B).astype(np.int32)
    for r in range(B):
        g[r, :g_len[r]] = rng.integers(0, 20, g_len[r])
        if rng.random() < 0.3 and g_len[r] > K:  # the n-gram chain contains the model chain
            g[r, :K] = d[r]
    conf = rng.choice([0.5, 0.9, 0.95, 1.0, 0.7], (B, K)).astype(np.float32)
    n = rng.integers(0, 17, B).astype(np.int32)
    n[rng.random(B) < 0.3] = 15
    a = rng.integers(0, 2, B).astype(np.int32)
    m = np.maximum(n, rng.integers(0, 400, B)).astype(np.int32)
    return [d, conf, rng.integers(0, K + 1, B).astype(np.int32), g, g_len, n, a, m]


@pytest.mark.gpu
@pytest.mark.parametrize("coef", ["table5", "constant"])
def test_static_pricing_at_the_arrays_full_size(S, coef):
    """256 requests x 31 slots (every word of the key area), budgets near the
    slot count, twice in a row against the workspace call."""
    rng = np.random.default_rng(256)
    B, K, L = 256, 7, 31
    arrays = _random_inputs(rng, B, K, L)
    est = S.EstimatorTable(W.table5_coef() if coef == "table5" else W.constant_coef(0.9), L)
    ws = S.Workspace(B, 1, K, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for budget in (B * L - 3, B * L, B * L + 7):
        common = (0.04, budget, L, "proposed", True)
        ref = _run(S, False, est, arrays, *common, ws=ws)
        for _ in range(2):
            _equal(_run(S, True, est, arrays, *common, status=status), ref)
    assert int(status.item()) == 0 and ws.status() == 0


@pytest.mark.gpu
def test_static_pricing_allocates_nothing(S):
    """After a warm-up call, further calls change neither torch's allocated
    bytes nor the device's free memory."""
    c = W.mixed_bs128()
    arrays = [torch.as_tensor(np.ascontiguousarray(x)).cuda() for x in _inputs(c)]
    d, conf, d_len, g, g_len, n, a, m = arrays
    B, L = g.shape
    est = S.EstimatorTable(c["coef"], c["L"])
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = (torch.empty((B, L), **i32), torch.empty((B, L), device="cuda"), torch.empty(B, **i32),
            torch.empty(B, **i32), torch.empty(B, **i32), torch.empty(B + 1, **i32),
            torch.empty((B, L), dtype=torch.uint8, device="cuda"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        S.spec_price_and_allocate_static(d, conf, d_len, g, g_len, n, a, m, est, c["lam"], c["budget"],
                                         c["max_verify_len"], c["policy"], c["draft_greedy"], *outs,
                                         status_word=status)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(8):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(status.item()) == 0
