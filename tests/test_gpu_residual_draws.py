"""Draws from max(0, p - q) after a rejected drafted token (the second launch
of sampled chain verification, one CTA per (request, chunk)).  These cases
load the draw path -- many rejected requests, invalid requests beside valid
ones, both element types, a vocabulary above 2^18 -- and check the draws
against the oracle, a clean status, and that the call leaves the workspace's
per-request counters and draw-record flags at zero for the next call."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from ._gpu import compare_sampled, gpu_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S
    S.build()
    return S


def _left_at_zero(ws, B):
    """the arrival counters, the draw counters and the draw records' flags of the first B requests"""
    off = ws.struct.base - ws.buf.data_ptr()
    raw = ws.buf[off:off + ws.struct.bytes].cpu().numpy()
    c1 = raw[ws.struct.off_counter:ws.struct.off_counter + 4 * B].view(np.uint32)
    c2 = raw[ws.struct.off_counter2:ws.struct.off_counter2 + 4 * B].view(np.uint32)
    flags = raw[ws.struct.off_record:ws.struct.off_record + 64 * B].reshape(B, 64)[:, :4].copy().view(np.int32)
    return not c1.any() and not c2.any() and not flags.any()


def _random_round(rng, B, L, K, V, ell_max, dtype):
    ell = rng.integers(1, ell_max + 1, B).astype(np.int32)
    ro = np.concatenate([[0], np.cumsum(ell + 1)]).astype(np.int32)
    z = (rng.standard_normal((int(ro[-1]), V)) * 2).astype(np.float32)
    draft = (rng.standard_normal((B, K, V)) * 2).astype(np.float32)
    chain = rng.integers(0, V, (B, L)).astype(np.int32)
    for r in range(B):  # drafts from the draft rows' argmax: accepted often enough to reach later positions
        for i in range(min(K, int(ell[r]))):
            if rng.random() < 0.6:
                chain[r, i] = int(draft[r, i].argmax())
    pm = np.ones((B, L), np.uint8)
    pm[:, :K] = (rng.random((B, K)) < 0.8).astype(np.uint8) ^ 1  # most positions carry a draft distribution
    if dtype == "bf16":
        z, draft = W.bf16_bits(z), W.bf16_bits(draft)
    return z, ro, chain, ell, pm, draft


@pytest.mark.parametrize("V,dtype", [(32000, "bf16"), (20000, "f32"), (151936, "bf16"), (151936, "f32"),
                                     (300000, "f32")])
def test_many_rejections(S, V, dtype):
    rng = np.random.default_rng(V + 7)
    B, L, K = (64, 8, 6) if V < 100000 else (24, 8, 6) if V < 200000 else (6, 5, 4)
    z, ro, chain, ell, pm, draft = _random_round(rng, B, L, K, V, L, dtype)
    ws = S.Workspace(B, int(ro[-1]), K, V)
    rejected = 0
    for step in range(5):
        g = gpu_chain(S, ws, z, ro, chain, ell, pm, draft, 1.0, seed=9, step=step)
        o = O.verify_chain(z, ro, chain, ell, pm, draft, 1.0, 9, step)
        compare_sampled(g, o, z, ro, chain, ell, pm, draft, 1.0)
        rejected += int(sum(1 for r in range(B) if o.n_accepted[r] < ell[r] and pm[r, o.n_accepted[r]] == 0))
        assert ws.status() == 0
        assert _left_at_zero(ws, B)
    # most requests end in a draw from max(0, p - q)
    assert rejected > 2 * B


def test_invalid_requests_beside_rejected_ones(S):
    rng = np.random.default_rng(3)
    B, L, K, V = 8, 7, 5, 4099
    z, ro, chain, ell, pm, draft = _random_round(rng, B, L, K, V, L, "bf16")
    ell = ell.copy()
    ell[2] = L + 2  # longer than the chain
    ell[5] = int(ro[6] - ro[5])  # no bonus row left
    bad = (2, 5)
    ws = S.Workspace(B, int(ro[-1]), K, V)
    for step in range(3):
        ws.reset_status()
        g = gpu_chain(S, ws, z, ro, chain, ell, pm, draft, 1.0, seed=2, step=step)
        assert ws.status() == S.DEV_BITS["bad_length"]
        for r in bad:
            assert g["na"][r] == 0 and g["ne"][r] == 0 and np.all(g["out"][r] == -1)
        o = O.verify_chain(z, ro, chain, ell, pm, draft, 1.0, 2, step)
        # the valid requests one by one, each on its own rows
        for r in range(B):
            if r in bad:
                continue
            one = {k: v[r:r + 1] for k, v in g.items()}
            o1 = type("O1", (), {})()
            for k in ("u", "ratio", "n_accepted", "n_emitted", "out_tokens", "resid", "Z", "t"):
                setattr(o1, k, getattr(o, k)[r:r + 1])
            rows = np.arange(ro[r], ro[r + 1])
            compare_sampled(one, o1, z[rows], np.array([0, len(rows)], np.int32), chain[r:r + 1], ell[r:r + 1],
                            pm[r:r + 1], draft[r:r + 1], 1.0)
        assert _left_at_zero(ws, B)
