"""The ORACLE for one hybrid speculative-decoding round: numpy front end.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The product package never imports this module, and this module
never imports the product package: the two share no code.

The arithmetic lives in ``spec_oracle.c`` (plain single-threaded C, fp64
except where a value decides an integer that must match bit for bit); this
file only builds that library with gcc and marshals numpy arrays into it.
Sources, cited by title and section in the C file:
  * Hybrid Spark: Adaptive Speculative Decoding That Lets the Content Choose
    the Drafter (n-gram lookup, Eq. (1) estimator, chain value Eq. (3),
    contains rule, adaptive-verification allocation, lossless policies);
  * AdaSpark: Adaptive DSpark with Online Learning for Tree Verification and
    N-gram Fill (greedy tree verification, sec. 2.2; the candidate tree and
    its best-first order, sec. 3.1, sec. 3.3 Eq. (6));
  * Efficient speculative decoding with a fixed-cost parallel drafter
    (accept / resample rule, r accepted => r + 1 tokens);
  * Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (Philox).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspec_oracle.so")

POLICY = {"proposed": 0, "ngram_first": 1, "extension": 2, "model_only": 3, "ngram_only": 4}
SRC_MODEL, SRC_NGRAM, SRC_CONTAINS, SRC_EXTENSION = 0, 1, 2, 3
ST_BAD_TOKEN, ST_NONFINITE, ST_BAD_TREE, ST_BAD_LENGTH, ST_BAD_VALUE = 0x1, 0x2, 0x4, 0x8, 0x10


def build(force: bool = False) -> str:
    """Compile spec_oracle.c with gcc (no FMA contraction) into libspec_oracle.so."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "spec_oracle.h"))
    ):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         "-Wall", "-o", tmp, _SRC, "-lm"]
    )
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


class Estimator(C.Structure):
    _fields_ = [
        ("beta", C.c_double * 32),
        ("w_first", C.c_double), ("w_rest", C.c_double), ("delta", C.c_double),
        ("ell_first", C.c_double), ("ell_rest", C.c_double),
        ("kappa_first", C.c_double), ("kappa_rest", C.c_double),
        ("n_ref", C.c_int32), ("n_full", C.c_int32), ("m_cap", C.c_int32), ("m_ref", C.c_int32),
        ("use_constant_h", C.c_int32), ("pad_", C.c_int32),
        ("constant_h", C.c_double),
    ]


def make_estimator(coef: dict) -> Estimator:
    """coef: {'beta': [...], 'w_first':..., ..., 'n_ref', 'n_full', 'm_cap', 'm_ref',
    'constant_h' (optional)}."""
    e = Estimator()
    beta = list(coef.get("beta", []))
    for i, b in enumerate(beta):
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


_i32p = C.POINTER(C.c_int32)
_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_u8p = C.POINTER(C.c_uint8)
_u32p = C.POINTER(C.c_uint32)


def _declare(L):
    L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
    L.oracle_philox4x32_10.restype = None
    L.oracle_u01.argtypes = [C.c_uint32]
    L.oracle_u01.restype = C.c_double
    L.oracle_round_uniforms.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, _f64p, _f64p]
    L.oracle_round_uniforms.restype = None
    L.oracle_ngram_propose.argtypes = [_i32p, C.c_int64, _i32p, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_int32, C.c_int32, _i32p, _i32p, _i32p, _i32p, _i32p]
    L.oracle_ngram_propose.restype = C.c_int
    L.oracle_estimate_h.argtypes = [C.POINTER(Estimator), C.c_int32, C.c_int32, C.c_int32, C.c_int32]
    L.oracle_estimate_h.restype = C.c_float
    L.oracle_chain_value.argtypes = [_f32p, C.c_int32, C.c_float]
    L.oracle_chain_value.restype = C.c_float
    L.oracle_price_and_allocate.argtypes = [
        C.c_int32, C.c_int32, C.c_int32, _i32p, _f32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p,
        C.POINTER(Estimator), C.c_float, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
        _i32p, _f32p, _i32p, _i32p, _i32p, _i32p, _u8p]
    L.oracle_price_and_allocate.restype = C.c_int
    L.oracle_verify_chain.argtypes = [
        C.c_int32, C.c_int32, C.c_int32, C.c_void_p, _i32p, C.c_void_p, C.c_int32,
        _i32p, C.c_int32, _i32p, _u8p, C.c_double, C.c_uint64, C.c_uint64, _f64p,
        _i32p, _i32p, _i32p, _f64p, _f64p, _f64p, _i32p, _f64p, _f64p]
    L.oracle_verify_chain.restype = C.c_int
    L.oracle_residual_row.argtypes = [
        C.c_int32, C.c_int32, C.c_void_p, _i32p, C.c_void_p, C.c_int32, _i32p, C.c_int32, _u8p,
        C.c_double, C.c_int32, C.c_int32, C.c_int32, _f64p]
    L.oracle_residual_row.restype = C.c_int
    L.oracle_verify_tree.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_void_p, _i32p, _i32p,
                                     _i32p, C.c_int32, _i32p, _i32p, _i32p]
    L.oracle_verify_tree.restype = C.c_int
    L.oracle_row_argmax.argtypes = [C.c_void_p, C.c_int32, C.c_int32]
    L.oracle_row_argmax.restype = C.c_int32
    L.oracle_build_tree.argtypes = [C.c_int32, C.c_int32, C.c_int32, _i32p, _i32p, _f32p, _i32p, C.c_int32,
                                    C.c_int32, _i32p, _f32p, _f32p, C.c_int32, _i32p, _i32p, _i32p, _i32p, _f64p]
    L.oracle_ngram_fill.argtypes = [_i32p, C.c_int64, _i32p, C.c_int32, C.c_int32, C.c_int32, _i32p, C.c_int32,
                                    C.c_int32, C.c_int32, C.c_int32, _i32p, _i32p, _i32p]
    L.oracle_ngram_fill.restype = C.c_int
    L.oracle_build_tree.restype = C.c_int
    L.oracle_size_budget.argtypes = [C.c_int32, C.c_int32, _f32p, _i32p, C.c_int32, C.c_double, C.c_double,
                                     _i32p, _f64p, _f64p]
    L.oracle_size_budget.restype = C.c_int
    L.oracle_sample_drafts.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_double,
                                       C.c_uint64, C.c_uint64, _f64p, _i32p, _f64p, _f64p]
    L.oracle_sample_drafts.restype = C.c_int


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _logits(a):
    """-> (contiguous array, dtype code): float32 -> 0, bf16 bits (uint16) -> 1."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {a.dtype}")


def _check(st):
    if st < 0:
        raise ValueError("oracle rejected an argument")
    return int(st)


# --------------------------------------------------------------------------- philox
def philox4x32_10(ctr, key):
    c = (C.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (C.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (C.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def u01(w: int) -> float:
    return float(lib().oracle_u01(int(w) & 0xFFFFFFFF))


def round_uniforms(seed: int, step: int, r: int, i: int):
    u, u2 = C.c_double(), C.c_double()
    lib().oracle_round_uniforms(int(seed), int(step), int(r), int(i), C.byref(u), C.byref(u2))
    return u.value, u2.value


# --------------------------------------------------------------------------- A1
@dataclass
class NgramOut:
    g: np.ndarray
    g_len: np.ndarray
    match_n: np.ndarray
    agree: np.ndarray
    copy_len: np.ndarray
    status: int


def ngram_propose(hist, hist_len, n_min, n_max, max_propose=15, copy_cap=256) -> NgramOut:
    hist = _c(hist, np.int32)
    hist_len = _c(hist_len, np.int32)
    B, stride = hist.shape
    g = np.empty((B, max_propose), np.int32)
    g_len, n, a, m = (np.empty(B, np.int32) for _ in range(4))
    st = lib().oracle_ngram_propose(_p(hist, C.c_int32), stride, _p(hist_len, C.c_int32), B,
                                    n_min, n_max, max_propose, copy_cap, _p(g, C.c_int32),
                                    _p(g_len, C.c_int32), _p(n, C.c_int32), _p(a, C.c_int32),
                                    _p(m, C.c_int32))
    return NgramOut(g, g_len, n, a, m, _check(st))


# --------------------------------------------------------------------------- A2
def estimate_h(coef, k, n, a, m) -> np.float32:
    e = make_estimator(coef)
    return np.float32(lib().oracle_estimate_h(C.byref(e), k, n, a, m))


def chain_value(S, lam) -> np.float32:
    S = _c(S, np.float32)
    return np.float32(lib().oracle_chain_value(_p(S, C.c_float), len(S), np.float32(lam)))


@dataclass
class PriceOut:
    chain: np.ndarray
    S: np.ndarray
    chain_len: np.ndarray
    source: np.ndarray
    verify_len: np.ndarray
    row_off: np.ndarray
    point_mass: np.ndarray
    status: int


def price_and_allocate(d, c, d_len, g, g_len, match_n, agree, copy_len, coef, lam, budget,
                       max_verify_len, policy="proposed", draft_greedy=True) -> PriceOut:
    d = _c(d, np.int32)
    c = _c(c, np.float32)
    g = _c(g, np.int32)
    B, K = d.shape
    L = g.shape[1]
    d_len, g_len, match_n, agree, copy_len = (_c(v, np.int32) for v in (d_len, g_len, match_n, agree, copy_len))
    e = make_estimator(coef)
    chain = np.empty((B, L), np.int32)
    S = np.empty((B, L), np.float32)
    chain_len, source, verify_len = (np.empty(B, np.int32) for _ in range(3))
    row_off = np.empty(B + 1, np.int32)
    pm = np.empty((B, L), np.uint8)
    pol = POLICY[policy] if isinstance(policy, str) else int(policy)
    st = lib().oracle_price_and_allocate(
        B, K, L, _p(d, C.c_int32), _p(c, C.c_float), _p(d_len, C.c_int32), _p(g, C.c_int32),
        _p(g_len, C.c_int32), _p(match_n, C.c_int32), _p(agree, C.c_int32), _p(copy_len, C.c_int32),
        C.byref(e), np.float32(lam), int(budget), int(max_verify_len), pol, 1 if draft_greedy else 0,
        _p(chain, C.c_int32), _p(S, C.c_float), _p(chain_len, C.c_int32), _p(source, C.c_int32),
        _p(verify_len, C.c_int32), _p(row_off, C.c_int32), _p(pm, C.c_uint8))
    return PriceOut(chain, S, chain_len, source, verify_len, row_off, pm, _check(st))


# --------------------------------------------------------------------------- A3
@dataclass
class VerifyOut:
    out_tokens: np.ndarray
    n_accepted: np.ndarray
    n_emitted: np.ndarray
    ratio: np.ndarray
    u: np.ndarray
    resid: np.ndarray
    pos: np.ndarray
    t: np.ndarray
    Z: np.ndarray
    status: int


def verify_chain(target_logits, row_off, chain, verify_len, point_mass=None, draft_logits=None,
                 temperature=0.0, seed=0, step=0, u_override=None) -> VerifyOut:
    """target_logits: [rows, V] float32 or bf16 bits (uint16); draft_logits: [B, K, V] or None."""
    tl, dt = _logits(target_logits)
    V = tl.shape[-1]
    chain = _c(chain, np.int32)
    B, L = chain.shape
    row_off = _c(row_off, np.int32)
    verify_len = _c(verify_len, np.int32)
    pm = None if point_mass is None else _c(point_mass, np.uint8)
    if draft_logits is not None:
        dl, dt2 = _logits(draft_logits)
        assert dt2 == dt and dl.shape[-1] == V
        K = dl.shape[1]
    else:
        dl, K = None, 0
    uo = None if u_override is None else _c(u_override, np.float64)
    out = np.empty((B, L + 1), np.int32)
    na, ne = np.empty(B, np.int32), np.empty(B, np.int32)
    ratio, u = np.empty((B, L)), np.empty((B, L))
    resid, t, Z = np.empty(B), np.empty(B), np.empty(B)
    pos = np.empty(B, np.int32)
    st = lib().oracle_verify_chain(
        B, V, dt, tl.ctypes.data, _p(row_off, C.c_int32), None if dl is None else dl.ctypes.data, K,
        _p(chain, C.c_int32), L, _p(verify_len, C.c_int32), None if pm is None else _p(pm, C.c_uint8),
        float(temperature), int(seed), int(step), None if uo is None else _p(uo, C.c_double),
        _p(out, C.c_int32), _p(na, C.c_int32), _p(ne, C.c_int32), _p(ratio, C.c_double),
        _p(u, C.c_double), _p(resid, C.c_double), _p(pos, C.c_int32), _p(t, C.c_double), _p(Z, C.c_double))
    return VerifyOut(out, na, ne, ratio, u, resid, pos, t, Z, _check(st))


def residual_row(target_logits, row_off, chain, r, i, rejected, point_mass=None, draft_logits=None,
                 temperature=1.0) -> np.ndarray:
    tl, dt = _logits(target_logits)
    V = tl.shape[-1]
    chain = _c(chain, np.int32)
    L = chain.shape[1]
    row_off = _c(row_off, np.int32)
    pm = None if point_mass is None else _c(point_mass, np.uint8)
    dl, K = (None, 0) if draft_logits is None else (_logits(draft_logits)[0], draft_logits.shape[1])
    out = np.empty(V)
    _check(lib().oracle_residual_row(V, dt, tl.ctypes.data, _p(row_off, C.c_int32),
                                     None if dl is None else dl.ctypes.data, K, _p(chain, C.c_int32), L,
                                     None if pm is None else _p(pm, C.c_uint8), float(temperature),
                                     int(r), int(i), int(rejected), _p(out, C.c_double)))
    return out


# --------------------------------------------------------------------------- A4
@dataclass
class TreeOut:
    path: np.ndarray
    accept_len: np.ndarray
    out_tokens: np.ndarray
    status: int


def verify_tree(logits, node_off, tok, parent, max_nodes) -> TreeOut:
    lg, dt = _logits(logits)
    V = lg.shape[-1]
    node_off = _c(node_off, np.int32)
    tok, parent = _c(tok, np.int32), _c(parent, np.int32)
    B = len(node_off) - 1
    path = np.empty((B, max_nodes), np.int32)
    out = np.empty((B, max_nodes), np.int32)
    al = np.empty(B, np.int32)
    st = lib().oracle_verify_tree(B, V, dt, lg.ctypes.data, _p(node_off, C.c_int32), _p(tok, C.c_int32),
                                  _p(parent, C.c_int32), int(max_nodes), _p(path, C.c_int32),
                                  _p(al, C.c_int32), _p(out, C.c_int32))
    return TreeOut(path, al, out, _check(st))


def row_argmax(row) -> int:
    a, dt = _logits(row)
    return int(lib().oracle_row_argmax(a.ctypes.data, a.shape[-1], dt))


# --------------------------------------------------------------------------- tree builder
@dataclass
class TreeBuild:
    tok: np.ndarray       # [B x width], -1 past n_rows
    parent: np.ndarray    # [B x width], local; -1 at the anchor and past n_rows
    cand_id: np.ndarray   # [B x width]
    n_rows: np.ndarray    # [B]
    Q: np.ndarray         # [B x (1 + P Kc + Lg)], -1 past the last candidate
    status: int


def build_tree(anchor, cand_tok, cand_score, ng_tok, ng_len, ng_score, ng_adj, width) -> TreeBuild:
    """ng_tok [B x Lg] with ng_len [B] (one chain, from the anchor), or
    [B x C x Lg] with ng_len [B x C] (chain 0 from the anchor, chain c from
    pick c-1)."""
    cand_tok, cand_score = _c(cand_tok, np.int32), _c(cand_score, np.float32)
    B, P, Kc = cand_tok.shape
    ng_tok = _c(ng_tok, np.int32)
    if ng_tok.ndim != 3:
        ng_tok = ng_tok.reshape(B, 1, -1)
    nc, Lg = ng_tok.shape[1], ng_tok.shape[2]
    anchor, ng_len = _c(anchor, np.int32), _c(ng_len, np.int32).reshape(B, nc)
    ng_score, ng_adj = _c(ng_score, np.float32), _c(ng_adj, np.float32)
    tok = np.empty((B, width), np.int32)
    parent = np.empty((B, width), np.int32)
    cid = np.empty((B, width), np.int32)
    nr = np.empty(B, np.int32)
    Q = np.empty((B, 1 + P * Kc + nc * Lg))
    st = lib().oracle_build_tree(B, P, Kc, _p(anchor, C.c_int32), _p(cand_tok, C.c_int32),
                                 _p(cand_score, C.c_float), _p(ng_tok, C.c_int32), nc, Lg, _p(ng_len, C.c_int32),
                                 _p(ng_score, C.c_float), _p(ng_adj, C.c_float), int(width), _p(tok, C.c_int32),
                                 _p(parent, C.c_int32), _p(cid, C.c_int32), _p(nr, C.c_int32),
                                 _p(Q, C.c_double))
    return TreeBuild(tok, parent, cid, nr, Q, _check(st))


@dataclass
class FillOut:
    tok: np.ndarray  # [B x (P+1) x Lg], -1 past each chain's end
    len: np.ndarray  # [B x (P+1)]
    ev: np.ndarray   # [B x (P+1) x Lg]: copy length (> 0) or minus the follower count
    status: int


def ngram_fill(hist, hist_len, cand_tok, n_min, copy_cap, max_depth, Lg) -> FillOut:
    """The n-gram chains of a candidate tree from the anchor and from each pick."""
    hist = _c(hist, np.int32)
    B, stride = hist.shape
    cand_tok = _c(cand_tok, np.int32)
    _, P, Kc = cand_tok.shape
    hist_len = _c(hist_len, np.int32)
    tok = np.empty((B, P + 1, Lg), np.int32)
    ln = np.empty((B, P + 1), np.int32)
    ev = np.empty((B, P + 1, Lg), np.int32)
    st = lib().oracle_ngram_fill(_p(hist, C.c_int32), stride, _p(hist_len, C.c_int32), B, P, Kc,
                                 _p(cand_tok, C.c_int32), int(n_min), int(copy_cap), int(max_depth), int(Lg),
                                 _p(tok, C.c_int32), _p(ln, C.c_int32), _p(ev, C.c_int32))
    return FillOut(tok, ln, ev, _check(st))


# --------------------------------------------------------------------------- budget sizing
@dataclass
class BudgetOut:
    b_star: int
    lam: float
    G: np.ndarray  # G(b) for b = 0..#slots


def size_budget(S, chain_len, max_verify_len, C0, p) -> BudgetOut:
    S = _c(S, np.float32)
    B, L = S.shape
    chain_len = _c(chain_len, np.int32)
    b = np.zeros(1, np.int32)
    lam = np.zeros(1)
    G = np.empty(B * L + 1)
    _check(lib().oracle_size_budget(B, L, _p(S, C.c_float), _p(chain_len, C.c_int32), int(max_verify_len),
                                    float(C0), float(p), _p(b, C.c_int32), _p(lam, C.c_double), _p(G, C.c_double)))
    n = int(np.minimum(np.minimum(chain_len, max_verify_len), L).clip(0).sum())
    return BudgetOut(int(b[0]), float(lam[0]), G[:n + 1])


# --------------------------------------------------------------------------- probabilistic drafting
@dataclass
class DraftOut:
    y: np.ndarray   # [B x K]
    u: np.ndarray   # [B x K] the uniforms
    q: np.ndarray   # [B x K] q of the drawn token (-1 for a flagged row)
    status: int


def sample_drafts(draft_logits, temperature, seed=0, step=0, u_override=None) -> DraftOut:
    """draft_logits [B x K x V] fp32, or bf16 bits (uint16)."""
    lg, dt = _logits(draft_logits)
    B, K, V = lg.shape
    y = np.empty((B, K), np.int32)
    u = np.empty((B, K))
    q = np.empty((B, K))
    uo = None if u_override is None else _c(u_override, np.float64)
    st = lib().oracle_sample_drafts(B, K, V, dt, lg.ctypes.data, float(temperature), int(seed), int(step),
                                    None if uo is None else _p(uo, C.c_double), _p(y, C.c_int32),
                                    _p(u, C.c_double), _p(q, C.c_double))
    return DraftOut(y, u, q, _check(st))
