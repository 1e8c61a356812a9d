"""One hybrid speculative-decoding round on preallocated device buffers.

ChainRound holds every buffer of steps 1-3 for one batch shape and launches
spec_draft_and_price (steps 1 and 2 in one kernel; or spec_ngram_propose then
spec_price_and_allocate) -> spec_verify_chain on one stream with no host
synchronisation in between (Hybrid Spark sec. 4.4: the host only passes lambda
and the budget as scalars).  The launches can be captured once into a CUDA
graph and replayed.
"""
from __future__ import annotations

import torch

from . import (EstimatorTable, Workspace, spec_draft_and_price, spec_ngram_propose,
               spec_price_and_allocate, spec_size_budget, spec_verify_chain)


class ChainRound:
    def __init__(self, B, stride, K, L, V, logits_dtype, max_rows, coef, n_min, n_max, copy_cap=256,
                 device="cuda", with_draft=False):
        i32 = dict(dtype=torch.int32, device=device)
        self.B, self.K, self.L, self.V, self.max_rows = B, K, L, V, max_rows
        self.n_min, self.n_max, self.copy_cap = n_min, n_max, copy_cap
        self.hist = torch.zeros((B, stride), **i32)
        self.hist_len = torch.zeros(B, **i32)
        self.d = torch.zeros((B, K), **i32)
        self.c = torch.zeros((B, K), dtype=torch.float32, device=device)
        self.d_len = torch.zeros(B, **i32)
        self.g = torch.zeros((B, L), **i32)
        self.g_len, self.match_n, self.agree, self.copy_len = (torch.zeros(B, **i32) for _ in range(4))
        self.chain = torch.zeros((B, L), **i32)
        self.S = torch.zeros((B, L), dtype=torch.float32, device=device)
        self.chain_len, self.source, self.verify_len = (torch.zeros(B, **i32) for _ in range(3))
        self.row_off = torch.zeros(B + 1, **i32)
        self.point_mass = torch.zeros((B, L), dtype=torch.uint8, device=device)
        self.out_tokens = torch.zeros((B, L + 1), **i32)
        self.n_accepted, self.n_emitted = torch.zeros(B, **i32), torch.zeros(B, **i32)
        self.logits = torch.zeros((max_rows, V), dtype=logits_dtype, device=device)
        self.draft_logits = torch.zeros((B, K, V), dtype=logits_dtype, device=device) if with_draft else None
        self.ws = Workspace(B, max_rows, K, V, device=device)
        self.est = EstimatorTable(coef, L, device=device)
        self.graph = None

    def load(self, hist, hist_len, d, c, d_len):
        self.hist.copy_(torch.as_tensor(hist), non_blocking=True)
        self.hist_len.copy_(torch.as_tensor(hist_len), non_blocking=True)
        self.d.copy_(torch.as_tensor(d), non_blocking=True)
        self.c.copy_(torch.as_tensor(c), non_blocking=True)
        self.d_len.copy_(torch.as_tensor(d_len), non_blocking=True)

    def draft_and_price(self, lam, budget, max_verify_len, policy="proposed", draft_greedy=True, stream=None,
                        fused=True):
        if fused:
            spec_draft_and_price(self.hist, self.hist_len, self.n_min, self.n_max, self.copy_cap, self.g,
                                 self.g_len, self.match_n, self.agree, self.copy_len, self.d, self.c, self.d_len,
                                 self.est, lam, budget, max_verify_len, policy, draft_greedy, self.chain, self.S,
                                 self.chain_len, self.source, self.verify_len, self.row_off, self.point_mass,
                                 self.ws, stream)
            return
        spec_ngram_propose(self.hist, self.hist_len, self.n_min, self.n_max, self.L, self.copy_cap, self.g,
                           self.g_len, self.match_n, self.agree, self.copy_len, self.ws, stream)
        spec_price_and_allocate(self.d, self.c, self.d_len, self.g, self.g_len, self.match_n, self.agree,
                                self.copy_len, self.est, lam, budget, max_verify_len, policy, draft_greedy,
                                self.chain, self.S, self.chain_len, self.source, self.verify_len,
                                self.row_off, self.point_mass, self.ws, stream)

    def verify(self, temperature=0.0, seed=0, step=0, row_off=None, stream=None, drafted=False):
        """drafted: the draft rows' statistics come from this round's
        spec_sample_drafts (spec_verify_chain_drafted)."""
        spec_verify_chain(self.logits, self.row_off if row_off is None else row_off, self.max_rows,
                          self.chain, self.verify_len, self.out_tokens, self.n_accepted, self.n_emitted,
                          self.ws, draft_logits=self.draft_logits,
                          point_mass=self.point_mass, temperature=temperature, seed=seed, step=step,
                          stream=stream, drafted=drafted)

    def run(self, lam, budget, max_verify_len, policy="proposed", draft_greedy=True, temperature=0.0,
            seed=0, step=0, stream=None):
        self.draft_and_price(lam, budget, max_verify_len, policy, draft_greedy, stream)
        self.verify(temperature, seed, step, stream=stream)

    def capture(self, **kw):
        """Capture run(**kw) into a CUDA graph (replay with .graph.replay())."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run(stream=s, **kw)  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(**kw)
        self.graph = g
        return g


class BudgetSizer:
    """Stale budget sizing (Hybrid Spark sec. 4.4, App. O): after the allocation
    of step t, spec_size_budget computes b* and lambda from step t's survivals
    on a side stream and copies them to pinned host memory; step t + 2 passes
    them to the pricing step as host scalars.  Steps 0 and 1 use the given
    initial values.  The next step's lookup waits for the sizing kernel (it
    overwrites the survivals the sizing reads), never for the host copy."""

    def __init__(self, C0, p, budget0, lam0, max_verify_len, device="cuda"):
        self.C0, self.p, self.mvl = float(C0), float(p), int(max_verify_len)
        self.dev_b = torch.zeros(2, dtype=torch.int32, device=device)
        self.dev_l = torch.zeros(2, dtype=torch.float32, device=device)
        self.host_b = torch.zeros(2, dtype=torch.int32).pin_memory()
        self.host_l = torch.zeros(2, dtype=torch.float32).pin_memory()
        self.copied = [None, None]
        self.sized = None
        self.init = (int(budget0), float(lam0))
        self.side = torch.cuda.Stream(device=device)
        self.ws = Workspace(1, 1, 1, 1, device=device)

    def params(self, step):
        """(budget, lambda) for `step`: sized from step - 2's survivals."""
        slot = step % 2
        ev = self.copied[slot]
        if step < 2 or ev is None:
            return self.init
        ev.synchronize()  # recorded two steps ago: normally long complete
        return int(self.host_b[slot]), float(self.host_l[slot])

    def size(self, rnd, step, stream=None):
        """Enqueue the sizing of `step`'s survivals (after its allocation on `stream`)."""
        stream = stream or torch.cuda.current_stream()
        slot = step % 2
        self.side.wait_stream(stream)
        with torch.cuda.stream(self.side):
            spec_size_budget(rnd.S, rnd.chain_len, self.mvl, self.C0, self.p, self.dev_b[slot:slot + 1],
                             self.dev_l[slot:slot + 1], self.ws, self.side)
            self.sized = torch.cuda.Event()
            self.sized.record(self.side)
            self.host_b[slot].copy_(self.dev_b[slot], non_blocking=True)
            self.host_l[slot].copy_(self.dev_l[slot], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.side)
            self.copied[slot] = ev

    def before_next_step(self, stream=None):
        """Order the next step's lookup after the sizing kernel that reads this
        step's survivals (a device-side wait)."""
        if self.sized is not None:
            (stream or torch.cuda.current_stream()).wait_event(self.sized)
