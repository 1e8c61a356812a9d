"""Seeded synthetic inputs for one hybrid speculative-decoding round.

This module is shared by both sides of the parity tests (the CUDA path and the
oracle) and by ``bench.py``.  It holds none of the round's arithmetic: it only
draws token histories, drafter chains, confidences and logits with the shapes,
sizes and structure of the workloads the pages measure on.  Random numbers the
method itself draws (the drafter's sampled tokens under probabilistic drafting)
are drawn here and passed in as inputs.

None of the pages' benchmark suites (NextCoder, EditBench, Blazedit, CanItEdit,
InstructCoder, MT-Bench, SPEED-Bench, Spec-Bench) is available; the generators
below stand in for their shapes only:
  * code editing: a Zipf(1.1) "program" followed by an edited copy of it,
    edits applied per span (geometric span lengths, mean 8) at a given rate;
  * chat: i.i.d. Zipf(1.1) text with no copy structure;
  * long context: Zipf text with repeated copied spans.
Token frequencies follow Zipf(1.1) over ranks 1..V mapped to ids by a seeded
permutation.  All seeds are NumPy PCG64.

Workload names and sizes:
  tiny      B=4,   V=1024,   history 512,   fp32 logits, 8 rows / request
  edit_bs4  B=4,   V=151936, history 2048,  bf16 logits (code editing)
  mixed_bs128 B=128, V=151936, context 4096, bf16 logits (half edit, half chat)
  tree_bs32 B=32,  V=151936, trees of 4/8/12/16 rows, bf16 logits
  long_bs64 B=64,  V=151936, history 32768, fp32 logits, 16 rows / request
"""
from __future__ import annotations

import functools

import numpy as np

# --------------------------------------------------------------------------
# Estimator coefficients, Hybrid Spark App. D, Table 5 (fit on the SPEED-Bench
# fitting half), and the reduced estimators of App. E, Table 7.  These are the
# pages' data; both sides receive them as inputs.
# --------------------------------------------------------------------------
_TABLE5 = {
    "qwen3_4b": ([-0.220, 0.155, 0.506, 0.683, 0.788, 0.697, 0.766, 0.721, 0.631, 0.658,
                  0.761, 0.803, 0.762, 0.862, 0.811],
                 (-0.0893, -0.0001, 1.2455, 1.1998, 0.1322, 2.0118, 1.8333)),
    "qwen3_8b": ([-0.414, -0.006, 0.246, 0.457, 0.551, 0.372, 0.613, 0.496, 0.501, 0.448,
                  0.516, 0.573, 0.554, 0.479, 0.744],
                 (-0.1301, 0.0303, 1.3938, 1.2694, -0.0385, 2.5317, 1.7287)),
    "gemma4_12b": ([-0.630, -0.227, -0.087, 0.086, 0.456, 0.263, 0.340, 0.541, 0.401, 0.443,
                    0.566, 0.678, 0.759, 0.779, 0.932],
                   (-0.0173, 0.0683, 1.1741, 1.1134, 0.1844, 2.1470, 1.5580)),
    "north_mini_code": ([-0.426, -0.204, -0.045, 0.044, 0.175, 0.084, -0.051, -0.137, -0.417,
                         -0.586, -0.582, -0.581, -0.478, -0.308, -0.154],
                        (-0.1422, -0.0757, 2.0234, 1.3238, 0.9809, 1.6695, 1.6321)),
    "llama3_1_8b": ([-0.070, 0.287, 0.544, 0.726, 0.950, 0.958, 0.897, -0.420, 0.607, 0.485,
                     0.602, 0.537, 0.611, 0.362, 0.762],
                    (-0.1248, 0.0233, 1.4169, 1.9266, 0.0714, 1.3100, 1.5100)),
}


def table5_coef(model: str = "qwen3_4b", n_full: int = 15) -> dict:
    beta, (wf, wr, de, lf, lr, kf, kr) = _TABLE5[model]
    return {"beta": list(beta), "w_first": wf, "w_rest": wr, "delta": de, "ell_first": lf,
            "ell_rest": lr, "kappa_first": kf, "kappa_rest": kr, "n_ref": 5, "n_full": n_full,
            "m_cap": 256, "m_ref": 15}


def table7_coef(estimator: int) -> dict:
    """Reduced estimators 1-5 (Hybrid Spark App. E, Table 7); a dash is a zero term.
    Estimators 3-5 share one coefficient between the first and later tokens."""
    rows = {
        1: ([2.117] * 15, None, None, None),
        2: ([1.158, 1.702, 2.104, 2.325, 2.466, 2.420, 2.536, 2.544, 2.515, 2.605, 2.757, 2.854,
             2.877, 3.036, 3.046], None, None, None),
        3: ([0.793, 1.293, 1.658, 1.845, 1.962, 1.882, 1.960, 1.923, 1.841, 1.876, 1.981, 2.025,
             1.992, 2.098, 2.053], 0.196, None, None),
        4: ([0.860, 1.345, 1.700, 1.880, 1.987, 1.897, 1.967, 1.922, 1.834, 1.859, 1.956, 1.994,
             1.950, 2.045, 1.988], None, 2.070, None),
        5: ([-0.247, 0.144, 0.495, 0.671, 0.776, 0.685, 0.754, 0.709, 0.618, 0.646, 0.749, 0.791,
             0.750, 0.850, 0.799], None, 2.014, 1.261),
    }
    beta, w, kappa, delta = rows[estimator]
    return {"beta": beta, "w_first": w or 0.0, "w_rest": w or 0.0, "delta": delta or 0.0,
            "ell_first": 0.0, "ell_rest": 0.0, "kappa_first": kappa or 0.0,
            "kappa_rest": kappa or 0.0, "n_ref": 5, "n_full": 15, "m_cap": 256, "m_ref": 15}


def constant_coef(h: float) -> dict:
    return {"constant_h": h, "n_ref": 5, "n_full": 15, "m_cap": 256, "m_ref": 15}


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    out = ((u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@functools.lru_cache(maxsize=8)
def _zipf_table(V: int, s: float, perm_seed: int):
    ranks = np.arange(1, V + 1, dtype=np.float64)
    w = ranks ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    perm = np.random.default_rng(perm_seed).permutation(V).astype(np.int32)
    return cdf, perm


def zipf_tokens(rng, n, V, s=1.1, perm_seed=7) -> np.ndarray:
    """n tokens, Zipf(s) over ranks 1..V, ranks mapped to ids by a seeded permutation."""
    cdf, perm = _zipf_table(int(V), float(s), int(perm_seed))
    idx = np.searchsorted(cdf, rng.random(int(n)), side="right")
    return perm[np.minimum(idx, V - 1)]


def edited_copy(rng, src, rate, V, mean_span=8.0) -> np.ndarray:
    """A copy of src whose spans (geometric lengths, mean 8) are each replaced, with
    probability `rate`, by a fresh Zipf span of geometric length."""
    out = []
    i = 0
    p = 1.0 / mean_span
    while i < len(src):
        span = int(rng.geometric(p))
        if rng.random() < rate:
            out.append(zipf_tokens(rng, int(rng.geometric(p)), V))
        else:
            out.append(src[i:i + span])
        i += span
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


def _pad_to(rng, a, n, V):
    if len(a) >= n:
        return a[:n]
    return np.concatenate([a, zipf_tokens(rng, n - len(a), V)]).astype(np.int32)


def _model_chain(rng, truth, conf, V):
    """A drafter chain: the true token with probability c_k, else a random other token."""
    B, K = conf.shape
    d = np.empty((B, K), np.int32)
    hit = rng.random((B, K)) < conf
    rand = zipf_tokens(rng, B * K, V).reshape(B, K)
    same = rand == truth[:, :K]
    rand[same] = (rand[same] + 1) % V
    d[:] = np.where(hit, truth[:, :K], rand)
    return d


def _draft_logits(rng, d_intended, V, scale=2.0, margin=6.0):
    """Draft logits N(0, 2) with a margin on the intended token (float32 [B, K, V])."""
    B, K = d_intended.shape
    z = rng.standard_normal((B, K, V), dtype=np.float32) * np.float32(scale)
    bi, ki = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    z[bi, ki, d_intended] += np.float32(margin)
    return z


def _sample_rows(rng, logits, T):
    """One token per row from softmax(logits / T) (the drafter's own sampling)."""
    z = logits.astype(np.float64) / T
    z -= z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    c = np.cumsum(p, axis=-1)
    u = rng.random(c.shape[:-1] + (1,))
    return np.minimum((c < u).sum(axis=-1), logits.shape[-1] - 1).astype(np.int32)


def truth_margin(V: int, T: float, p_target: float = 0.9, scale: float = 1.0) -> float:
    """Logit margin giving the planted token probability ~p_target under softmax(z / T)
    with N(0, scale^2) background logits (T = 0: a clear argmax)."""
    if T <= 0:
        return 8.0
    mass = V * np.exp(0.5 * scale * scale / (T * T))  # E[sum exp(z / T)] over the background
    return float(T * np.log(p_target / (1 - p_target) * mass))


def target_logits(rng, rows_truth, V, dtype, margin):
    """Target logits N(0, 1) with `margin` added on each row's true next token.
    rows_truth: int array [rows] (-1: no planted token).  dtype 'f32' or 'bf16'."""
    R = len(rows_truth)
    z = rng.standard_normal((R, V), dtype=np.float32)
    ok = rows_truth >= 0
    z[np.nonzero(ok)[0], rows_truth[ok]] += np.float32(margin)
    return z if dtype == "f32" else bf16_bits(z)


def rows_truth_for_layout(truth, row_off, verify_len, total_rows=None):
    """The true next token of every verify row of a compact (or strided) layout:
    row row_off[r] + i holds position i + 1 of request r, whose truth is truth[r, i]."""
    B = len(verify_len)
    total = int(row_off[B]) if total_rows is None else int(total_rows)
    out = np.full(total, -1, np.int32)
    for r in range(B):
        for i in range(int(verify_len[r]) + 1):
            out[int(row_off[r]) + i] = truth[r, i]
    return out


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
def tiny(seed=1000, probabilistic=False, temperature=1.0):
    """B=4, V=1024: a uniform 256-token program followed by a copy with 20% of
    positions replaced uniformly; n-gram match n in {1,2,3}, proposals up to 15;
    a 7-token model chain from fp32 draft logits N(0, 2); target logits = draft
    logits + N(0, 1) over 8 materialised rows per request; n-gram estimates
    h_k = 0.9 (survival 0.9^k); budget 24; lambda 0.04."""
    rng = np.random.default_rng(seed)
    B, V, K, L, stride = 4, 1024, 7, 15, 512
    hist = np.empty((B, stride), np.int32)
    hist_len = np.empty(B, np.int32)
    for r in range(B):
        prog = rng.integers(0, V, 256, dtype=np.int32)
        copy = prog.copy()
        sub = rng.random(256) < 0.2
        copy[sub] = rng.integers(0, V, int(sub.sum()), dtype=np.int32)
        hist[r] = np.concatenate([prog, copy])
        hist_len[r] = 256 + int(rng.integers(16, 256 - 32))
    draft = rng.standard_normal((B, K, V), dtype=np.float32) * np.float32(2.0)
    if probabilistic:
        d = _sample_rows(rng, draft, temperature)
    else:
        d = draft.argmax(axis=-1).astype(np.int32)
    rows = 8
    tl = np.empty((B * rows, V), np.float32)
    for r in range(B):
        tl[r * rows:r * rows + K] = draft[r] + rng.standard_normal((K, V), dtype=np.float32)
        tl[r * rows + K:(r + 1) * rows] = (rng.standard_normal((rows - K, V), dtype=np.float32) * 2
                                           + rng.standard_normal((rows - K, V), dtype=np.float32))
    return {
        "name": "tiny", "B": B, "V": V, "K": K, "L": L, "hist": hist, "hist_len": hist_len,
        "n_min": 1, "n_max": 3, "copy_cap": 256,
        "d": d, "c": rng.uniform(0.92, 0.96, (B, K)).astype(np.float32),
        "d_len": np.full(B, K, np.int32), "draft_logits": draft,
        "coef": constant_coef(0.9), "lam": 0.04, "budget": 24, "max_verify_len": rows - 1,
        "policy": "extension" if probabilistic else "proposed", "draft_greedy": not probabilistic,
        "temperature": temperature, "seed": 0, "dtype": "f32",
        "target_logits": tl, "rows_per_request": rows,
        "row_off_materialised": np.arange(B + 1, dtype=np.int32) * rows,
    }


def _edit_requests(rng, n, src_len, stride, rate, V, t_lo, t_hi, L):
    hist = np.empty((n, stride), np.int32)
    hist_len = np.empty(n, np.int32)
    for r in range(n):
        src = zipf_tokens(rng, src_len, V)
        rr = rate[r] if np.ndim(rate) else rate
        copy = edited_copy(rng, src, rr, V)
        hist[r] = _pad_to(rng, np.concatenate([src, copy]).astype(np.int32), stride, V)
        hist_len[r] = int(rng.integers(t_lo, t_hi))
        assert hist_len[r] + L + 1 <= stride
    return hist, hist_len


def edit_bs4(seed=1001, temperature=0.0, probabilistic=False, edit_rates=None):
    """Code editing at batch 4, V=151936, bf16: each request holds a 2048-token history,
    a Zipf(1.1) 1024-token source followed by its edited copy (edit rate per request
    from {0,15,30,45,60,70}%).  Model chain of 7 (true token with probability c_k,
    c_k ~ U[0.92, 0.96]) plus an n-gram chain up to 15; budget 64, lambda 0.04.
    Greedy drafting uses the proposed policy; probabilistic drafting (T=1) the
    extension policy, with the chain sampled from bf16 draft logits."""
    rng = np.random.default_rng(seed)
    B, V, K, L, stride = 4, 151936, 7, 15, 2048
    rates = np.asarray(edit_rates if edit_rates is not None else
                       rng.choice([0.0, 0.15, 0.30, 0.45, 0.60, 0.70], B))
    hist, hist_len = _edit_requests(rng, B, 1024, stride, rates, V, 1024 + 16, 2048 - 32, L)
    truth = np.stack([hist[r, hist_len[r]:hist_len[r] + L + 1] for r in range(B)])
    c = rng.uniform(0.92, 0.96, (B, K)).astype(np.float32)
    d_int = _model_chain(rng, truth, c, V)
    draft = None
    if probabilistic:
        draft_f = _draft_logits(rng, d_int, V, margin=truth_margin(V, temperature, 0.8, 2.0))
        draft_b = bf16_bits(draft_f)
        d = _sample_rows(rng, bf16_to_f32(draft_b), temperature)
        draft = draft_b
    else:
        d = d_int
    return {
        "name": "edit_bs4", "B": B, "V": V, "K": K, "L": L, "hist": hist, "hist_len": hist_len,
        "n_min": 5, "n_max": 15, "copy_cap": 256, "truth": truth, "edit_rates": rates,
        "d": d, "c": c, "d_len": np.full(B, K, np.int32), "draft_logits": draft,
        "coef": table5_coef("qwen3_4b"), "lam": 0.04, "budget": 64, "max_verify_len": L,
        "policy": "extension" if probabilistic else "proposed", "draft_greedy": not probabilistic,
        "temperature": temperature, "seed": 0, "dtype": "bf16",
        "margin": truth_margin(V, temperature),
    }


def mixed_bs128(seed=1002):
    """Batch 128, context ~4096 (current length in [3072, 4064] of a 4096-token buffer):
    64 code-edit requests (2048-token source + copy at 30% edit rate) and 64 chat
    requests (i.i.d. Zipf(1.1) text).  Budget 256 over both drafters' chains by price,
    lambda 0.3, T=0, bf16 V=151936 logits."""
    rng = np.random.default_rng(seed)
    B, V, K, L, stride = 128, 151936, 7, 15, 4096
    half = B // 2
    h_edit, l_edit = _edit_requests(rng, half, 2048, stride, 0.30, V, 3072, 4064, L)
    h_chat = zipf_tokens(rng, half * stride, V).reshape(half, stride)
    l_chat = rng.integers(3072, 4064, half).astype(np.int32)
    hist = np.concatenate([h_edit, h_chat]).astype(np.int32)
    hist_len = np.concatenate([l_edit, l_chat]).astype(np.int32)
    truth = np.stack([hist[r, hist_len[r]:hist_len[r] + L + 1] for r in range(B)])
    c = np.concatenate([rng.uniform(0.92, 0.96, (half, K)),
                        rng.uniform(0.69, 0.74, (half, K))]).astype(np.float32)
    d = _model_chain(rng, truth, c, V)
    return {
        "name": "mixed_bs128", "B": B, "V": V, "K": K, "L": L, "hist": hist, "hist_len": hist_len,
        "n_min": 5, "n_max": 15, "copy_cap": 256, "truth": truth,
        "d": d, "c": c, "d_len": np.full(B, K, np.int32), "draft_logits": None,
        "coef": table5_coef("qwen3_4b"), "lam": 0.3, "budget": 256, "max_verify_len": L,
        "policy": "proposed", "draft_greedy": True, "temperature": 0.0, "seed": 0,
        "dtype": "bf16", "margin": truth_margin(V, 0.0),
    }


def long_bs64(seed=1004, B=64, stride=32768):
    """Batch 64 x 32768-token Zipf histories, each holding one 512-token span and five
    later copies of it; the current suffix lies inside the last copy.  n-gram match
    n <= 4, proposals up to 15, budget 512, lambda 0.3; chain verification at T=0.7
    over fp32 V=151936 logits materialised as 16 rows per request; point-mass drafts."""
    rng = np.random.default_rng(seed)
    V, K, L, span = 151936, 7, 15, 512
    hist = zipf_tokens(rng, B * stride, V).reshape(B, stride).astype(np.int32)
    hist_len = np.empty(B, np.int32)
    for r in range(B):
        T = stride - 64
        src_at = int(rng.integers(0, stride // 8))
        src = hist[r, src_at:src_at + span].copy()
        last_at = T - int(rng.integers(span - 64, span - 31))  # copy ends 32..64 past T
        starts = sorted(rng.choice(np.arange(src_at + span, last_at - span, span), 4, replace=False))
        for s0 in list(starts) + [last_at]:
            hist[r, s0:s0 + span] = src
        hist_len[r] = T
    truth = np.stack([hist[r, hist_len[r]:hist_len[r] + L + 1] for r in range(B)])
    c = rng.uniform(0.69, 0.74, (B, K)).astype(np.float32)
    d = _model_chain(rng, truth, c, V)
    rows = L + 1
    return {
        "name": "long_bs64", "B": B, "V": V, "K": K, "L": L, "hist": hist, "hist_len": hist_len,
        "n_min": 1, "n_max": 4, "copy_cap": 256, "truth": truth,
        "d": d, "c": c, "d_len": np.full(B, K, np.int32), "draft_logits": None,
        "coef": table5_coef("qwen3_4b", n_full=4), "lam": 0.3, "budget": 512,
        "max_verify_len": L, "policy": "proposed", "draft_greedy": True, "temperature": 0.7,
        "seed": 0, "dtype": "f32", "margin": truth_margin(V, 0.7),
        "rows_per_request": rows,
        "row_off_materialised": np.arange(B + 1, dtype=np.int32) * rows,
    }


def materialised_logits(cfg, rng_seed=None):
    """Logits for a workload whose rows are materialised per request (rows_per_request
    rows at row_off = r * rows): row i of request r plants truth[r, i]."""
    rng = np.random.default_rng(cfg.get("seed_logits", 77) if rng_seed is None else rng_seed)
    B, rows = cfg["B"], cfg["rows_per_request"]
    rt = np.full(B * rows, -1, np.int32)
    for r in range(B):
        rt[r * rows:(r + 1) * rows] = cfg["truth"][r, :rows]
    return target_logits(rng, rt, cfg["V"], cfg["dtype"], cfg["margin"])


def compact_logits(cfg, row_off, verify_len, rng_seed=78):
    """Logits in the compact verify layout the allocation produced."""
    rng = np.random.default_rng(rng_seed)
    rt = rows_truth_for_layout(cfg["truth"], row_off, verify_len)
    return target_logits(rng, rt, cfg["V"], cfg["dtype"], cfg["margin"])


# --------------------------------------------------------------------------
# trees (AdaSpark sec. 2.2 shape, Fig. 1; order by Q = prod q, Prop. 1)
# --------------------------------------------------------------------------
def tree_blocks(seed=1003, B=32, P=8, Kc=4, V=151936):
    """Inputs of the candidate-tree builder for B requests: a block of P positions
    with Kc ranked candidates each (distinct tokens per position), scored with the
    shape of the acceptance model's prior on the tree-verification page (pick:
    ln 2 + logit h with the confidence head h ~ Beta(2, 2); sibling: log r with r
    its share of the siblings' total, r ~ Dirichlet(1)); a 4096-token Zipf history
    whose last 6 tokens repeat an earlier passage, and the 15 tokens that followed
    that passage as the n-gram chain from the anchor (scored 0: a source
    precision of 1/2, so no agreement adjustment)."""
    rng = np.random.default_rng(seed)
    anchor = np.empty(B, np.int32)
    cand_tok = np.empty((B, P, Kc), np.int32)
    cand_score = np.empty((B, P, Kc), np.float32)
    hist = np.empty((B, 4096), np.int32)
    ng_tok = np.empty((B, 15), np.int32)
    for r in range(B):
        h = zipf_tokens(rng, 4096, V)
        at = int(rng.integers(0, 2048))
        h[4096 - 6:] = h[at:at + 6]
        hist[r] = h
        ng_tok[r] = h[at + 6:at + 6 + 15]
        anchor[r] = h[-1]
        for i in range(P):
            toks = []
            while len(toks) < Kc:
                t = int(zipf_tokens(rng, 1, V)[0])
                if t not in toks:
                    toks.append(t)
            cand_tok[r, i] = toks
            hc = float(np.clip(rng.beta(2.0, 2.0), 1e-4, 1 - 1e-4))
            cand_score[r, i, 0] = np.log(2.0) + np.log(hc / (1 - hc))
            if Kc > 1:
                cand_score[r, i, 1:] = np.log(np.maximum(rng.dirichlet(np.ones(Kc - 1)), 1e-6))
    # a few requests follow the block with the chain, so that it agrees with picks
    for r in range(0, B, 4):
        ng_tok[r, :min(P, 15)] = cand_tok[r, :min(P, 15), 0]
    return {"B": B, "P": P, "Kc": Kc, "V": V, "anchor": anchor, "cand_tok": cand_tok, "cand_score": cand_score,
            "ng_tok": ng_tok, "ng_len": np.full(B, 15, np.int32), "ng_score": np.zeros(B, np.float32),
            "ng_adj": np.zeros(B, np.float32), "hist": hist}


def tree_fill_bs32(seed=1011, width=16, B=32, P=8, Kc=4, V=151936):
    """The tree round with its n-gram chains made by the fill from the request's
    own text: tree_blocks' 4096-token histories (their last 6 tokens repeat an
    earlier passage), with the drafter's picks following that passage's
    continuation in every fourth request and for its first three positions in
    the next one (so that chains agree with picks and chains from picks read
    on).  Fill parameters: copy length >= 4 for a passage (so that contexts
    matched only by their last three tokens take the follower rule), copies
    capped at 256, chains to 32 tokens below the anchor."""
    cfg = tree_blocks(seed=seed, B=B, P=P, Kc=Kc, V=V)
    hist = cfg["hist"]
    for r in range(B):
        # where the history's last 6 tokens occurred before (the planted repeat)
        tail = hist[r, -6:]
        at = next(a for a in range(4096 - 6) if np.array_equal(hist[r, a:a + 6], tail))
        follow = P if r % 4 == 0 else (3 if r % 4 == 1 else 0)
        for i in range(follow):
            t = int(hist[r, at + 6 + i])
            row = cfg["cand_tok"][r, i]
            if t in row[1:]:
                row[list(row).index(t)] = row[0]
            row[0] = t
    cfg.update({"name": f"tree_fill_bs32_w{width}", "width": width, "max_nodes": width, "dtype": "bf16",
                "hist_len": np.full(B, 4096, np.int32), "n_min": 4, "copy_cap": 256, "max_depth": 32,
                "Lg": 32, "ng_score": np.zeros(B, np.float32),
                "ng_adj": np.full(B, float(np.log(0.7 / 0.3)), np.float32)})
    return cfg


def flatten_trees(tok, parent, n_rows):
    """[B x width] tree rows (valid up to n_rows[r]) -> node_off [B + 1] and the
    rows of all requests back to back."""
    n_rows = np.asarray(n_rows, np.int64)
    node_off = np.concatenate([[0], np.cumsum(n_rows)]).astype(np.int32)
    t = np.concatenate([np.asarray(tok)[r, :n_rows[r]] for r in range(len(n_rows))]).astype(np.int32)
    p = np.concatenate([np.asarray(parent)[r, :n_rows[r]] for r in range(len(n_rows))]).astype(np.int32)
    return node_off, t, p


def _capped_geometric_rate(depth, mean):
    """alpha in [0, 1] with sum_{k=1..depth} alpha^k = min(mean, depth): the
    acceptance rate whose geometric accept length, capped at `depth`, has that
    mean (bisection; alpha = 1 when the cap is at or below the mean)."""
    if depth <= mean:
        return 1.0
    lo, hi = 0.0, 1.0
    for _ in range(60):
        a = 0.5 * (lo + hi)
        if sum(a ** k for k in range(1, depth + 1)) < mean:
            lo = a
        else:
            hi = a
    return 0.5 * (lo + hi)


def tree_logits(node_off, tok, parent, V, seed=1005, dtype="bf16", margin=8.0, mean_accept=3.0):
    """bf16 (or fp32) logits N(0, 1) for the rows of given trees, with a planted
    true path per request whose accept length has mean `mean_accept` (3),
    capped by the tree.

    Request r's accept length A is geometric on 0..d, d the depth of its tree
    (P(A >= k) = alpha^k for k <= d), with alpha chosen so that E[A] =
    min(3, d); the draws are stratified over the batch (request r takes the
    quantile at (pi(r) + v) / B for a seeded permutation pi and v ~ U[0, 1)),
    so that the batch's mean is close to the law's.  The path walks A steps
    from the anchor, each to a uniformly chosen child whose subtree is deep
    enough for the steps left (the spine of picks or an n-gram chain; siblings
    are leaves).  At each path node but the last the target's argmax is the
    token of the next path node (margin +margin); at the last node it is a
    token that matches none of its children.  Returns (logits, planted paths
    as row indices)."""
    rng = np.random.default_rng(seed)
    N = int(node_off[-1])
    B = len(node_off) - 1
    row_truth = np.full(N, -1, np.int32)
    planted = []
    strata = (rng.permutation(B) + rng.random(B)) / max(B, 1)
    for r in range(B):
        base, n = int(node_off[r]), int(node_off[r + 1] - node_off[r])
        kids_of = [[] for _ in range(n)]
        for j in range(1, n):
            kids_of[int(parent[base + j])].append(j)
        height = [0] * n  # parents precede children: one backward pass
        for j in range(n - 1, 0, -1):
            pj = int(parent[base + j])
            height[pj] = max(height[pj], height[j] + 1)
        d = height[0]
        alpha = _capped_geometric_rate(d, mean_accept)
        u = float(strata[r])
        A = d if alpha >= 1.0 else min(d, int(np.floor(np.log1p(-u) / np.log(alpha))))
        cur, depth, path = 0, 0, [0]
        while depth < A:
            pool = [j for j in kids_of[cur] if height[j] >= A - depth - 1]
            nxt = pool[int(rng.integers(0, len(pool)))]
            row_truth[base + cur] = tok[base + nxt]
            cur = nxt
            path.append(cur)
            depth += 1
        kid_toks = {int(tok[base + j]) for j in kids_of[cur]}
        t = int(rng.integers(0, V))
        while t in kid_toks:
            t = (t + 1) % V
        row_truth[base + cur] = t
        planted.append(path)
    return target_logits(rng, row_truth, V, dtype, margin), planted


def tree_bs32(seed=1003, width=16, B=32):
    """Greedy tree verification, batch 32: the builder inputs of tree_blocks (8
    picks with top-4 ranked candidates, confidences Beta(2,2), an n-gram chain
    from a planted repeat in a 4096-token history) and the tree width (4, 8, 12
    or 16 rows).  The tree itself comes from the builder; tree_logits plants a
    true path on it."""
    cfg = tree_blocks(seed=seed + 17 * width, B=B)
    cfg.update({"name": f"tree_bs32_w{width}", "width": width, "max_nodes": width, "dtype": "bf16"})
    return cfg
