"""spec_verify_chain_drafted: verification that takes the draft rows'
per-chunk statistics and the logits at the drawn tokens from the preceding
spec_sample_drafts on the same workspace, instead of reading the draft rows
again.  Its results must equal spec_verify_chain's bit for bit on the same
round (that call is the one checked against the oracle), whatever the
workspace's row capacity (the drafting call places the draft rows' slots after
it, the plain call after its own row bound)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from ._gpu import compare_sampled, gpu_chain, logits_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S
    S.build()
    return S


def _round(S, c, T, seed, step, extra_rows):
    """Draw the drafts on the device, price with them as the model chain, and
    lay out the target rows: the inputs of one probabilistic round."""
    B, K, V = c["B"], c["K"], c["V"]
    ws = S.Workspace(B, B * (c["L"] + 1) + extra_rows, K, V)
    dt = logits_dev(c["draft_logits"])
    y = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    S.spec_sample_drafts(dt, T, y, ws, seed=seed, step=step)
    d = y.cpu().numpy()
    ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
    lay = O.price_and_allocate(d, c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                               c["coef"], c["lam"], c["budget"], c["max_verify_len"], c["policy"], False)
    return ws, dt, lay


@pytest.mark.parametrize("rate", [0.0, 0.30, 0.70])
@pytest.mark.parametrize("extra_rows", [0, 37])
def test_drafted_verification_equals_the_plain_call(S, rate, extra_rows):
    c = W.edit_bs4(temperature=1.0, probabilistic=True, edit_rates=[rate] * 4)
    T = 1.0
    for step in range(4):
        ws, dt, lay = _round(S, c, T, seed=11, step=step, extra_rows=extra_rows)
        logits = W.compact_logits(c, lay.row_off, lay.verify_len)
        lt = logits_dev(logits)
        args = (S, ws, None, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, c["draft_logits"], T)
        g1 = gpu_chain(*args, seed=5, step=step, logits_t=lt, draft_t=dt, drafted=True)  # right after drafting
        g0 = gpu_chain(*args, seed=5, step=step, logits_t=lt, draft_t=dt)
        for k in ("out", "na", "ne", "ratio", "u", "resid"):
            assert np.array_equal(g1[k], g0[k]), (k, step)
        o = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, c["draft_logits"], T,
                           5, step)
        compare_sampled(g1, o, logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass,
                        c["draft_logits"], T)
        assert ws.status() == 0


def test_drafted_verification_flags_another_temperature(S):
    c = W.edit_bs4(temperature=1.0, probabilistic=True, edit_rates=[0.3] * 4)
    ws, dt, lay = _round(S, c, 1.0, seed=1, step=0, extra_rows=0)
    logits = W.compact_logits(c, lay.row_off, lay.verify_len)
    assert int((lay.point_mass[:, :c["K"]] == 0).sum()) > 0  # some positions carry a draft distribution
    gpu_chain(S, ws, logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, c["draft_logits"], 0.9,
              seed=1, step=0, draft_t=dt, drafted=True)
    assert ws.status() & S.DEV_BITS["bad_value"]
