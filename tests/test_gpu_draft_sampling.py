"""GPU parity of probabilistic drafting (spec_sample_drafts) against the
oracle.  Exactness: the uniforms bit-exact; the drawn token equal to the
oracle's, or valid under the oracle's CDF of q within 1e-5 (the kernel's
exponentials are fp32); q of the drawn token within 1e-5 absolute."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

from ._gpu import logits_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    S.load()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return S


def _gpu(S, z, T, seed, step, ws=None):
    B, K, V = z.shape
    ws = ws or S.Workspace(B, 1, K, V)
    y = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    u = torch.full((B, K), -7.0, device="cuda")
    q = torch.full((B, K), -7.0, device="cuda")
    S.spec_sample_drafts(logits_dev(z), T, y, ws, seed=seed, step=step, dbg_u=u, dbg_q=q)
    torch.cuda.synchronize()
    return y.cpu().numpy(), u.cpu().numpy(), q.cpu().numpy(), ws


def _q_rows(z, T):
    zf = W.bf16_to_f32(z) if z.dtype == np.uint16 else z
    x = zf.astype(np.float64) / T
    x -= x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def _compare(z, T, g_y, g_u, g_q, o, tol=1e-5):
    q = _q_rows(z, T)
    B, K = g_y.shape
    equal = 0
    for r in range(B):
        for k in range(K):
            assert g_u[r, k] == np.float32(o.u[r, k]), (r, k)
            y = int(g_y[r, k])
            assert 0 <= y < q.shape[-1]
            cdf = np.cumsum(q[r, k])
            lo = cdf[y - 1] if y > 0 else 0.0
            u = o.u[r, k]
            assert lo <= u + tol and cdf[y] >= u - tol, (r, k, y, int(o.y[r, k]), lo, cdf[y], u)
            assert abs(g_q[r, k] - q[r, k, y]) < tol
            equal += y == o.y[r, k]
    return equal


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_draft_sampling_on_the_code_editing_workload(S, T):
    c = W.edit_bs4(temperature=1.0, probabilistic=True)
    z = c["draft_logits"]  # bf16 bits [4 x 7 x 151936]
    ws = None
    total = equal = 0
    for step in range(4):
        y, u, q, ws = _gpu(S, z, T, 3, step, ws)
        o = O.sample_drafts(z, T, seed=3, step=step)
        equal += _compare(z, T, y, u, q, o)
        total += y.size
    assert equal >= total - 1
    assert ws.status() == 0


@pytest.mark.parametrize("V,dtype", [(2049, "f32"), (1000, "bf16"), (8, "f32"), (4097, "bf16"), (151936, "f32")])
def test_draft_sampling_ragged_vocab(S, V, dtype):
    rng = np.random.default_rng(V)
    z = (rng.standard_normal((3, 5, V)) * 2).astype(np.float32)
    if dtype == "bf16":
        z = W.bf16_bits(z)
    for step in range(3):
        y, u, q, ws = _gpu(S, z, 0.9, 5, step)
        _compare(z, 0.9, y, u, q, O.sample_drafts(z, 0.9, seed=5, step=step))
        assert ws.status() == 0


def test_draft_sampling_follows_q(S):
    rng = np.random.default_rng(9)
    z = (rng.standard_normal((2, 3, 8)) * 1.5).astype(np.float32)
    N = 1500
    counts = np.zeros((2, 3, 8))
    ws = None
    for step in range(N):
        y, _, _, ws = _gpu(S, z, 0.8, 2, step, ws)
        for r in range(2):
            for k in range(3):
                counts[r, k, y[r, k]] += 1
    q = _q_rows(z, 0.8)
    chi2 = ((counts - N * q) ** 2 / (N * q)).sum(axis=-1)
    assert np.all(chi2 < 30.0), chi2


def test_draft_sampling_flags_nonfinite_rows(S):
    z = np.zeros((2, 2, 64), np.float32)
    z[1, 0, 5] = np.nan
    y, _, _, ws = _gpu(S, z, 1.0, 0, 0)
    assert ws.status() & S.DEV_BITS["nonfinite"]
