"""GB300 (sm_103a) hot path of one hybrid speculative-decoding round.

A thin binding over the C ABI in ``include/spec.h`` (libspecgb.so, built in
tree by ``build()``): every function below only marshals torch tensors into
device pointers and forwards to the entry point of the same name, on the
current CUDA stream.  Every step of the round runs in the library's CUDA
kernels; there is no CPU path.  If the library is missing, every call raises.

Steps (see include/spec.h for the full contract of each):
  spec_ngram_propose       n-gram prompt lookup (Hybrid Spark sec. 4.1-4.2)
  spec_price_and_allocate  Eq. (1)-(3), contains rule, budget allocation
  spec_verify_chain        rejection-sampling / greedy chain verification
  spec_verify_tree         greedy tree verification (AdaSpark sec. 2.2)
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from ._build import LIB as _LIB_PATH
from ._build import build

__all__ = [
    "build", "load", "Workspace", "EstimatorTable", "SpecError", "spec_ngram_propose",
    "spec_price_and_allocate", "spec_price_and_allocate_static", "spec_draft_and_price", "spec_verify_chain", "spec_verify_chain_drafted", "spec_verify_tree", "spec_build_tree", "spec_ngram_fill", "spec_size_budget", "spec_sample_drafts", "POLICY",
    "DEV_BITS",
]

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_CUDA, SPEC_ERR_UNSUPPORTED, SPEC_ERR_WORKSPACE = 0, 1, 2, 3, 4
SPEC_F32, SPEC_BF16 = 0, 1
POLICY = {"proposed": 0, "ngram_first": 1, "extension": 2, "model_only": 3, "ngram_only": 4}
DEV_BITS = {"bad_token": 0x1, "nonfinite": 0x2, "bad_tree": 0x4, "bad_length": 0x8,
            "bad_value": 0x10, "timeout": 0x20, "overflow": 0x40}


class SpecError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn}: {msg} (status {code})")
        self.code = code


class WorkspaceStruct(C.Structure):
    _fields_ = [
        ("base", C.c_void_p), ("bytes", C.c_size_t),
        ("max_batch", C.c_int32), ("max_rows", C.c_int32), ("K", C.c_int32), ("vocab", C.c_int32),
        ("off_counter", C.c_size_t), ("off_counter2", C.c_size_t), ("off_record", C.c_size_t),
        ("off_rowkey", C.c_size_t), ("off_partial", C.c_size_t), ("off_partial2", C.c_size_t),
        ("off_keys", C.c_size_t), ("off_counter3", C.c_size_t), ("units", C.c_int32), ("pad_", C.c_int32),
    ]


class EstimatorStruct(C.Structure):
    _fields_ = [
        ("beta", C.c_double * 32),
        ("w_first", C.c_double), ("w_rest", C.c_double), ("delta", C.c_double),
        ("ell_first", C.c_double), ("ell_rest", C.c_double),
        ("kappa_first", C.c_double), ("kappa_rest", C.c_double),
        ("n_ref", C.c_int32), ("n_full", C.c_int32), ("m_cap", C.c_int32), ("m_ref", C.c_int32),
        ("use_constant_h", C.c_int32), ("pad_", C.c_int32),
        ("constant_h", C.c_double),
    ]


_lib = None
_vp, _i32, _i64, _f32, _u64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_uint64, C.c_size_t
_WSP = C.POINTER(WorkspaceStruct)
_ESTP = C.POINTER(EstimatorStruct)

SIGNATURES = {
    "spec_status_string": ([_i32], C.c_char_p),
    "spec_version": ([], _i32),
    "spec_workspace_bytes": ([_i32, _i32, _i32, _i32], _sz),
    "spec_workspace_init": ([_WSP, _vp, _sz, _i32, _i32, _i32, _i32, _vp], _i32),
    "spec_workspace_status_word": ([_WSP], _vp),
    "spec_estimator_table_bytes": ([_ESTP, _i32], _sz),
    "spec_estimator_build": ([_ESTP, _i32, _vp, _sz, _vp], _i32),
    "spec_ngram_propose": ([_vp, _i64, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                            _WSP, _vp], _i32),
    "spec_price_and_allocate": ([_i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ESTP, _vp,
                                 _sz, _f32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _WSP, _vp], _i32),
    "spec_price_and_allocate_static": ([_i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ESTP, _vp,
                                        _sz, _f32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _vp], _i32),
    "spec_draft_and_price": ([_vp, _i64, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                              _vp, _vp, _vp, _ESTP, _vp, _sz, _f32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                              _vp, _vp, _vp, _vp, _WSP, _vp], _i32),
    "spec_verify_chain": ([_i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _f32,
                           _u64, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _WSP, _vp], _i32),
    "spec_verify_chain_drafted": ([_i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _i32, _vp, _vp, _f32,
                                   _u64, _u64, _vp, _vp, _vp, _vp, _vp, _vp, _WSP, _vp], _i32),
    "spec_build_tree": ([_i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _vp,
                         _vp, _WSP, _vp], _i32),
    "spec_ngram_fill": ([_vp, _i64, _vp, _i32, _i32, _i32, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _WSP, _vp],
                        _i32),
    "spec_size_budget": ([_i32, _i32, _vp, _vp, _i32, C.c_double, C.c_double, _vp, _vp, _WSP, _vp], _i32),
    "spec_sample_drafts": ([_i32, _i32, _i32, _i32, _vp, _f32, _u64, _u64, _vp, _vp, _vp, _WSP, _vp], _i32),
    "spec_verify_tree": ([_i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _WSP, _vp],
                         _i32),
}


def load(path: str | None = None):
    """Load libspecgb.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(speculative_decoding_draft_spec_gb300.build())")
    lib = C.CDLL(p)
    for name, (argt, rest) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = rest
    if path is None:
        _lib = lib
    return lib


def _check(fn, code):
    if code != SPEC_OK:
        raise SpecError(fn, code, load().spec_status_string(code).decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


class Workspace:
    """Device workspace (status word, arrival counters, per-row partials) laid out
    for up to max_batch requests, max_rows logit rows, K draft rows per request
    and `vocab` entries per row.  The device memory comes from PyTorch."""

    def __init__(self, max_batch, max_rows, K, vocab, device="cuda", stream=None):
        lib = load()
        n = lib.spec_workspace_bytes(max_batch, max_rows, K, vocab)
        if n == 0:
            raise ValueError("invalid workspace capacity")
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        off = (-base) % 256
        self.struct = WorkspaceStruct()
        _check("spec_workspace_init",
               lib.spec_workspace_init(C.byref(self.struct), base + off, n, max_batch, max_rows, K, vocab,
                                       _stream(stream)))
        self.status_view = self.buf[off:off + 4].view(torch.int32)

    def status(self) -> int:
        """The device status word (synchronises: for tests and diagnostics)."""
        return int(self.status_view.item()) & 0xFFFFFFFF

    def reset_status(self):
        self.status_view.zero_()

    @property
    def ref(self):
        return C.byref(self.struct)


def make_estimator(coef: dict) -> EstimatorStruct:
    e = EstimatorStruct()
    for i, b in enumerate(coef.get("beta", [])):
        e.beta[i] = float(b)
    for name in ("w_first", "w_rest", "delta", "ell_first", "ell_rest", "kappa_first", "kappa_rest"):
        setattr(e, name, float(coef.get(name, 0.0)))
    e.n_ref = int(coef.get("n_ref", 5))
    e.n_full = int(coef.get("n_full", 15))
    e.m_cap = int(coef.get("m_cap", 256))
    e.m_ref = int(coef.get("m_ref", 15))
    if coef.get("constant_h") is not None:
        e.use_constant_h = 1
        e.constant_h = float(coef["constant_h"])
    return e


class EstimatorTable:
    """Eq. (1) tabulated on the GPU (fp64, rounded once to fp32) for chains of L."""

    def __init__(self, coef: dict, L: int, device="cuda", stream=None):
        lib = load()
        self.est = make_estimator(coef)
        self.L = L
        n = lib.spec_estimator_table_bytes(C.byref(self.est), L)
        if n == 0:
            raise ValueError("invalid estimator")
        self.table = torch.empty(n // 4, dtype=torch.float32, device=device)
        _check("spec_estimator_build",
               lib.spec_estimator_build(C.byref(self.est), L, _ptr(self.table), n, _stream(stream)))


def spec_ngram_propose(hist, hist_len, n_min, n_max, max_propose, copy_cap, g, g_len, match_n, agree,
                       copy_len, ws: Workspace, stream=None):
    B, stride = hist.shape
    _check("spec_ngram_propose", load().spec_ngram_propose(
        _ptr(hist), stride, _ptr(hist_len), B, n_min, n_max, max_propose, copy_cap, _ptr(g), _ptr(g_len),
        _ptr(match_n), _ptr(agree), _ptr(copy_len), ws.ref, _stream(stream)))


def spec_price_and_allocate(d, c, d_len, g, g_len, match_n, agree, copy_len, est: EstimatorTable, lam,
                            budget, max_verify_len, policy, draft_greedy, chain, S, chain_len, source,
                            verify_len, row_off, point_mass, ws: Workspace, stream=None):
    B, K = d.shape
    L = g.shape[1]
    pol = POLICY[policy] if isinstance(policy, str) else int(policy)
    _check("spec_price_and_allocate", load().spec_price_and_allocate(
        B, K, L, _ptr(d), _ptr(c), _ptr(d_len), _ptr(g), _ptr(g_len), _ptr(match_n), _ptr(agree),
        _ptr(copy_len), C.byref(est.est), _ptr(est.table), est.table.numel() * 4, float(lam), int(budget), int(max_verify_len),
        pol, 1 if draft_greedy else 0, _ptr(chain), _ptr(S), _ptr(chain_len), _ptr(source),
        _ptr(verify_len), _ptr(row_off), _ptr(point_mass), ws.ref, _stream(stream)))


def spec_price_and_allocate_static(d, c, d_len, g, g_len, match_n, agree, copy_len, est: EstimatorTable, lam,
                                   budget, max_verify_len, policy, draft_greedy, chain, S, chain_len, source,
                                   verify_len, row_off, point_mass, status_word=None, stream=None):
    """spec_price_and_allocate with its scratch in the library's fixed device
    array instead of a workspace (nothing is allocated; batch <= 256; calls
    that may overlap on one device race).  status_word: optional int32 device
    tensor of one element that receives the device error bits."""
    B, K = d.shape
    L = g.shape[1]
    pol = POLICY[policy] if isinstance(policy, str) else int(policy)
    _check("spec_price_and_allocate_static", load().spec_price_and_allocate_static(
        B, K, L, _ptr(d), _ptr(c), _ptr(d_len), _ptr(g), _ptr(g_len), _ptr(match_n), _ptr(agree),
        _ptr(copy_len), C.byref(est.est), _ptr(est.table), est.table.numel() * 4, float(lam), int(budget),
        int(max_verify_len), pol, 1 if draft_greedy else 0, _ptr(chain), _ptr(S), _ptr(chain_len), _ptr(source),
        _ptr(verify_len), _ptr(row_off), _ptr(point_mass), _ptr(status_word), _stream(stream)))


def spec_draft_and_price(hist, hist_len, n_min, n_max, copy_cap, g, g_len, match_n, agree, copy_len, d, c,
                         d_len, est: EstimatorTable, lam, budget, max_verify_len, policy, draft_greedy, chain, S,
                         chain_len, source, verify_len, row_off, point_mass, ws: Workspace, stream=None):
    B, stride = hist.shape
    K = d.shape[1]
    L = g.shape[1]
    pol = POLICY[policy] if isinstance(policy, str) else int(policy)
    _check("spec_draft_and_price", load().spec_draft_and_price(
        _ptr(hist), stride, _ptr(hist_len), B, n_min, n_max, copy_cap, _ptr(g), _ptr(g_len), _ptr(match_n),
        _ptr(agree), _ptr(copy_len), K, L, _ptr(d), _ptr(c), _ptr(d_len), C.byref(est.est), _ptr(est.table),
        est.table.numel() * 4, float(lam), int(budget), int(max_verify_len), pol, 1 if draft_greedy else 0,
        _ptr(chain), _ptr(S), _ptr(chain_len), _ptr(source), _ptr(verify_len), _ptr(row_off), _ptr(point_mass),
        ws.ref, _stream(stream)))


def spec_verify_chain(target_logits, row_off, max_rows, chain, verify_len, out_tokens, n_accepted,
                      n_emitted, ws: Workspace, draft_logits=None, point_mass=None, temperature=0.0,
                      seed=0, step=0, dbg_ratio=None, dbg_u=None, dbg_resid=None, stream=None, drafted=False):
    """drafted=True calls spec_verify_chain_drafted (the draft rows' statistics
    from the preceding spec_sample_drafts on this workspace)."""
    B, L = chain.shape
    V = target_logits.shape[-1]
    K = 0 if draft_logits is None else draft_logits.shape[1]
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise TypeError("draft and target logits must share a dtype")
    name = "spec_verify_chain_drafted" if drafted else "spec_verify_chain"
    _check(name, getattr(load(), name)(
        B, V, _dtype_code(target_logits), _ptr(target_logits), _ptr(row_off), int(max_rows),
        _ptr(draft_logits), K, _ptr(chain), L, _ptr(verify_len), _ptr(point_mass), float(temperature),
        int(seed), int(step), _ptr(out_tokens), _ptr(n_accepted), _ptr(n_emitted), _ptr(dbg_ratio),
        _ptr(dbg_u), _ptr(dbg_resid), ws.ref, _stream(stream)))


def spec_verify_chain_drafted(*args, **kw):
    """spec_verify_chain with the draft rows' statistics from spec_sample_drafts."""
    return spec_verify_chain(*args, drafted=True, **kw)


def spec_verify_tree(logits, node_off, max_rows, tok, parent, max_nodes, path, accept_len, out_tokens,
                     ws: Workspace, stream=None):
    B = node_off.shape[0] - 1
    V = logits.shape[-1]
    _check("spec_verify_tree", load().spec_verify_tree(
        B, V, _dtype_code(logits), _ptr(logits), _ptr(node_off), int(max_rows), _ptr(tok), _ptr(parent),
        int(max_nodes), _ptr(path), _ptr(accept_len), _ptr(out_tokens), ws.ref, _stream(stream)))


def spec_build_tree(anchor, cand_tok, cand_score, ng_tok, ng_len, ng_score, ng_adj, width, tok, parent, cand_id,
                    n_rows, ws: Workspace, stream=None):
    """cand_tok / cand_score [B x P x Kc]; ng_tok [B x Lg] with ng_len [B] (one
    chain, from the anchor) or [B x C x Lg] with ng_len [B x C] (chain 0 from
    the anchor, chain c from pick c-1); outputs tok / parent / cand_id
    [B x width], n_rows [B] (all int32 device tensors)."""
    B, P, Kc = cand_tok.shape
    nc, Lg = (ng_tok.shape[1], ng_tok.shape[2]) if ng_tok.dim() == 3 else (1, ng_tok.shape[1])
    _check("spec_build_tree", load().spec_build_tree(
        B, P, Kc, _ptr(anchor), _ptr(cand_tok), _ptr(cand_score), _ptr(ng_tok), nc, Lg, _ptr(ng_len),
        _ptr(ng_score), _ptr(ng_adj), int(width), _ptr(tok), _ptr(parent), _ptr(cand_id), _ptr(n_rows), ws.ref,
        _stream(stream)))


def spec_ngram_fill(hist, hist_len, cand_tok, n_min, copy_cap, max_depth, ng_tok, ng_len, ng_ev, ws: Workspace,
                    stream=None):
    """The n-gram chains of a candidate tree from the anchor and from each pick:
    hist [B x stride], hist_len [B], cand_tok [B x P x Kc]; outputs ng_tok /
    ng_ev [B x (P+1) x Lg], ng_len [B x (P+1)] (all int32 device tensors)."""
    B, stride = hist.shape
    P, Kc = cand_tok.shape[1], cand_tok.shape[2]
    Lg = ng_tok.shape[2]
    _check("spec_ngram_fill", load().spec_ngram_fill(
        _ptr(hist), stride, _ptr(hist_len), B, P, Kc, _ptr(cand_tok), int(n_min), int(copy_cap), int(max_depth), Lg,
        _ptr(ng_tok), _ptr(ng_len), _ptr(ng_ev), ws.ref, _stream(stream)))


def spec_size_budget(S, chain_len, max_verify_len, C0, p, out_budget, out_lambda, ws: Workspace, stream=None):
    """b* and lambda for a later step from survivals S [B x L] (device); out_budget:
    int32 device tensor of one element, out_lambda: float32 device tensor of one."""
    B, L = S.shape
    _check("spec_size_budget", load().spec_size_budget(
        B, L, _ptr(S), _ptr(chain_len), int(max_verify_len), float(C0), float(p), _ptr(out_budget),
        _ptr(out_lambda), ws.ref, _stream(stream)))


def spec_sample_drafts(draft_logits, temperature, y, ws: Workspace, seed=0, step=0, dbg_u=None, dbg_q=None,
                       stream=None):
    """y [B x K] ~ softmax(draft_logits [B x K x V] / T) per position (device tensors)."""
    B, K, V = draft_logits.shape
    _check("spec_sample_drafts", load().spec_sample_drafts(
        B, K, V, _dtype_code(draft_logits), _ptr(draft_logits), float(temperature), int(seed), int(step), _ptr(y),
        _ptr(dbg_u), _ptr(dbg_q), ws.ref, _stream(stream)))
