"""Helpers for the GPU parity tests: run each step through the C ABI on
device tensors, and compare sampled outputs with the oracle under the stated
exactness rules."""
import numpy as np
import torch

import oracle as O
import workloads as W

DEV = "cuda"


def dev(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


def logits_dev(a):
    """numpy float32 or bf16 bits (uint16) -> device float32 / bfloat16 tensor"""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def gpu_ngram(S, ws, hist, hist_len, n_min, n_max, L=15, cap=256):
    B = hist.shape[0]
    i32 = dict(dtype=torch.int32, device=DEV)
    g = torch.full((B, L), -7, **i32)
    out = [torch.full((B,), -7, **i32) for _ in range(4)]
    S.spec_ngram_propose(dev(hist, torch.int32), dev(hist_len, torch.int32), n_min, n_max, L, cap, g, *out, ws)
    torch.cuda.synchronize()
    return host(g), *[host(t) for t in out]


def gpu_price(S, ws, est, d, c, d_len, g, g_len, n, a, m, lam, budget, mvl, policy, greedy):
    B, K = d.shape
    L = g.shape[1]
    i32 = dict(dtype=torch.int32, device=DEV)
    chain = torch.full((B, L), -7, **i32)
    Sv = torch.full((B, L), -7.0, dtype=torch.float32, device=DEV)
    chain_len, source, verify_len = (torch.full((B,), -7, **i32) for _ in range(3))
    row_off = torch.full((B + 1,), -7, **i32)
    pm = torch.full((B, L), 7, dtype=torch.uint8, device=DEV)
    S.spec_price_and_allocate(dev(d, torch.int32), dev(c, torch.float32), dev(d_len, torch.int32),
                              dev(g, torch.int32), dev(g_len, torch.int32), dev(n, torch.int32),
                              dev(a, torch.int32), dev(m, torch.int32), est, lam, budget, mvl, policy, greedy,
                              chain, Sv, chain_len, source, verify_len, row_off, pm, ws)
    torch.cuda.synchronize()
    return dict(chain=host(chain), S=host(Sv), chain_len=host(chain_len), source=host(source),
                verify_len=host(verify_len), row_off=host(row_off), point_mass=host(pm))


def gpu_chain(S, ws, logits, row_off, chain, verify_len, pm=None, draft=None, T=0.0, seed=0, step=0,
              logits_t=None, draft_t=None, drafted=False):
    B, L = chain.shape
    i32 = dict(dtype=torch.int32, device=DEV)
    out = torch.full((B, L + 1), -7, **i32)
    na, ne = torch.full((B,), -7, **i32), torch.full((B,), -7, **i32)
    ratio = torch.full((B, L), -7.0, device=DEV)
    u = torch.full((B, L), -7.0, device=DEV)
    resid = torch.full((B,), -7.0, device=DEV)
    lt = logits_t if logits_t is not None else logits_dev(logits)
    dt = draft_t if draft_t is not None else (None if draft is None else logits_dev(draft))
    max_rows = int(row_off[-1])
    S.spec_verify_chain(lt, dev(row_off, torch.int32), max_rows, dev(chain, torch.int32),
                        dev(verify_len, torch.int32), out, na, ne, ws, draft_logits=dt,
                        point_mass=None if pm is None else dev(pm, torch.uint8), temperature=T, seed=seed,
                        step=step, dbg_ratio=ratio, dbg_u=u, dbg_resid=resid, drafted=drafted)
    torch.cuda.synchronize()
    return dict(out=host(out), na=host(na), ne=host(ne), ratio=host(ratio), u=host(u), resid=host(resid))


def gpu_tree(S, ws, logits, node_off, tok, parent, max_nodes, logits_t=None):
    B = len(node_off) - 1
    i32 = dict(dtype=torch.int32, device=DEV)
    path = torch.full((B, max_nodes), -7, **i32)
    out = torch.full((B, max_nodes), -7, **i32)
    al = torch.full((B,), -7, **i32)
    lt = logits_t if logits_t is not None else logits_dev(logits)
    S.spec_verify_tree(lt, dev(node_off, torch.int32), int(node_off[-1]), dev(tok, torch.int32),
                       dev(parent, torch.int32), max_nodes, path, al, out, ws)
    torch.cuda.synchronize()
    return dict(path=host(path), accept_len=host(al), out=host(out))


def compare_sampled(g, o, logits, row_off, chain, verify_len, pm, draft, T, tol=1e-5):
    """Exactness rules for T > 0: accept decisions bit-exact except where
    |u - min(1, ratio)| < tol (the request is not compared after such a point);
    a drawn id equal to the oracle's, or valid under the oracle's residual CDF
    within tol * Z of the oracle's threshold; its residual probability within
    tol absolute.  Returns counters for reporting."""
    B, L = chain.shape
    stats = dict(requests=B, exact=0, band=0, draw_equal=0, draw_band=0)
    for r in range(B):
        ell = int(verify_len[r])
        diverged = False
        for i in range(1, ell + 1):
            uo, ro = o.u[r, i - 1], o.ratio[r, i - 1]
            if uo < 0:
                break
            acc_o = ro >= 1.0 or uo < ro
            gr, gu = g["ratio"][r, i - 1], g["u"][r, i - 1]
            assert gu == np.float32(uo), (r, i, gu, uo)  # identical Philox uniforms
            acc_g = gr >= 1.0 or gu < gr
            if acc_o != acc_g:
                assert abs(uo - min(1.0, ro)) < tol, (r, i, uo, ro, gr)
                diverged = True
                stats["band"] += 1
                break
            if not acc_o:
                break
        if diverged:
            continue
        assert g["na"][r] == o.n_accepted[r] and g["ne"][r] == o.n_emitted[r], r
        n = int(o.n_accepted[r])
        assert np.array_equal(g["out"][r, :n], o.out_tokens[r, :n]), r
        assert np.all(g["out"][r, n + 1:] == -1)
        xg, xo = int(g["out"][r, n]), int(o.out_tokens[r, n])
        if xg == xo:
            stats["draw_equal"] += 1
            assert abs(g["resid"][r] - o.resid[r]) < tol, (r, g["resid"][r], o.resid[r])
        else:
            rejected = n < ell
            w = O.residual_row(logits, row_off, chain, r, n + 1, rejected, pm, draft, T)
            cdf = np.cumsum(w)
            Z, t = o.Z[r], o.t[r]
            before = cdf[xg - 1] if xg > 0 else 0.0
            assert before <= t + tol * Z and cdf[xg] >= t - tol * Z, (r, xg, xo, before, cdf[xg], t)
            assert abs(g["resid"][r] - w[xg] / Z) < tol
            stats["draw_band"] += 1
        stats["exact"] += 1
    return stats


def gpu_draft_price(S, ws, est, hist, hist_len, n_min, n_max, cap, d, c, d_len, lam, budget, mvl, policy, greedy,
                    L=15):
    """the fused steps 1 + 2 through spec_draft_and_price"""
    B, K = d.shape
    i32 = dict(dtype=torch.int32, device=DEV)
    g = torch.full((B, L), -7, **i32)
    gl, n, a, m = (torch.full((B,), -7, **i32) for _ in range(4))
    chain = torch.full((B, L), -7, **i32)
    Sv = torch.full((B, L), -7.0, dtype=torch.float32, device=DEV)
    chain_len, source, verify_len = (torch.full((B,), -7, **i32) for _ in range(3))
    row_off = torch.full((B + 1,), -7, **i32)
    pm = torch.full((B, L), 7, dtype=torch.uint8, device=DEV)
    S.spec_draft_and_price(dev(hist, torch.int32), dev(hist_len, torch.int32), n_min, n_max, cap, g, gl, n, a, m,
                           dev(d, torch.int32), dev(c, torch.float32), dev(d_len, torch.int32), est, lam, budget, mvl,
                           policy, greedy, chain, Sv, chain_len, source, verify_len, row_off, pm, ws)
    torch.cuda.synchronize()
    return dict(g=host(g), g_len=host(gl), match_n=host(n), agree=host(a), copy_len=host(m), chain=host(chain),
                S=host(Sv), chain_len=host(chain_len), source=host(source), verify_len=host(verify_len),
                row_off=host(row_off), point_mass=host(pm))


def gpu_build_tree(S, ws, anchor, cand_tok, cand_score, ng_tok, ng_len, ng_score, ng_adj, width):
    B = len(anchor)
    i32 = dict(dtype=torch.int32, device=DEV)
    tok, parent, cid = (torch.full((B, width), -7, **i32) for _ in range(3))
    nr = torch.full((B,), -7, **i32)
    S.spec_build_tree(dev(anchor, torch.int32), dev(cand_tok, torch.int32), dev(cand_score, torch.float32),
                      dev(np.asarray(ng_tok) if np.ndim(ng_tok) == 3 else np.asarray(ng_tok).reshape(B, -1),
                          torch.int32), dev(ng_len, torch.int32),
                      dev(ng_score, torch.float32), dev(ng_adj, torch.float32), width, tok, parent, cid, nr, ws)
    torch.cuda.synchronize()
    return dict(tok=host(tok), parent=host(parent), cand_id=host(cid), n_rows=host(nr))


def gpu_ngram_fill(S, ws, hist, hist_len, cand_tok, n_min, copy_cap, max_depth, Lg):
    B = len(hist_len)
    P = np.shape(cand_tok)[1]
    i32 = dict(dtype=torch.int32, device=DEV)
    tok, ev = (torch.full((B, P + 1, Lg), -7, **i32) for _ in range(2))
    ln = torch.full((B, P + 1), -7, **i32)
    S.spec_ngram_fill(dev(hist, torch.int32), dev(hist_len, torch.int32), dev(cand_tok, torch.int32), n_min,
                      copy_cap, max_depth, tok, ln, ev, ws)
    torch.cuda.synchronize()
    return dict(tok=host(tok), len=host(ln), ev=host(ev))


def assert_tree_equal(g, o, rel=1e-12):
    """The built trees equal the oracle's, except where the oracle's Q has a
    near-tie (relative gap <= rel) at the selection cut: there the two
    selections may differ among the tied candidates, and the GPU's must still
    be a tree of the same size whose sum of Q is within rel of the oracle's."""
    for r in range(len(o.n_rows)):
        n = int(o.n_rows[r])
        assert int(g["n_rows"][r]) == n, r
        if np.array_equal(g["cand_id"][r], o.cand_id[r]):
            assert np.array_equal(g["tok"][r], o.tok[r]) and np.array_equal(g["parent"][r], o.parent[r]), r
            continue
        Q = o.Q[r]
        sel_o, sel_g = set(o.cand_id[r, 1:n]), set(g["cand_id"][r, 1:n])
        diff = sel_o ^ sel_g
        cut = min(Q[list(sel_o)]) if sel_o else 1.0
        assert all(abs(Q[c] - cut) <= rel * cut for c in diff), (r, sorted(diff))
        assert abs(sum(Q[list(sel_g)]) - sum(Q[list(sel_o)])) <= rel * max(1.0, sum(Q[list(sel_o)])), r
        # the GPU's rows still form a depth-first layout, and a candidate that
        # both select has the same token under the same parent candidate
        gc, gp, gt = g["cand_id"][r], g["parent"][r], g["tok"][r]
        assert int(gc[0]) == 0 and int(gp[0]) == -1, r
        assert all(0 <= int(gp[i]) < i for i in range(1, n)), r
        o_tok = {int(o.cand_id[r, i]): int(o.tok[r, i]) for i in range(n)}
        o_par = {int(o.cand_id[r, i]): int(o.cand_id[r, int(o.parent[r, i])]) for i in range(1, n)}
        for i in range(1, n):
            c = int(gc[i])
            if c in o_par:
                assert int(gt[i]) == o_tok[c] and int(gc[int(gp[i])]) == o_par[c], (r, c)
