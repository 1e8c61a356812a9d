"""The C-ABI library builds, loads without a GPU, exports every entry point that
include/spec.h declares, and rejects bad arguments on the host before any
CUDA call (host-side fault injection: nothing here touches a GPU)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec.h")


@pytest.fixture(scope="module")
def spec():
    import speculative_decoding_draft_spec_gb300 as S

    S.build()
    return S


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", txt)))


def test_header_declares_the_four_steps():
    names = _declared()
    for step in ("spec_ngram_propose", "spec_price_and_allocate", "spec_verify_chain", "spec_verify_tree"):
        assert step in names


def test_library_exports_every_declared_symbol(spec):
    lib = spec.load()
    out = subprocess.run(["nm", "-D", "--defined-only", spec._build.LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (spec_[a-z_0-9]+)\b", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)


def test_binding_covers_every_declared_symbol(spec):
    assert set(_declared()) == set(spec.SIGNATURES)


def test_struct_layouts_match_the_header(spec):
    # sizes of the host structs as the C compiler lays them out
    src = ('#include "spec.h"\n#include <stdio.h>\n#include <stddef.h>\n'
           'int main(){printf("%zu %zu %zu %zu\\n", sizeof(spec_workspace), sizeof(spec_estimator),'
           ' offsetof(spec_workspace, units), offsetof(spec_estimator, constant_h));}')
    exe = os.path.join(ROOT, "_build", "layout_probe")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    with open(exe + ".c", "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                           "-o", exe, exe + ".c"])
    ws, est, ws_units, est_ch = map(int, subprocess.check_output([exe]).split())
    assert C.sizeof(spec.WorkspaceStruct) == ws
    assert C.sizeof(spec.EstimatorStruct) == est
    assert spec.WorkspaceStruct.units.offset == ws_units
    assert spec.EstimatorStruct.constant_h.offset == est_ch


def test_status_strings_and_version(spec):
    lib = spec.load()
    assert lib.spec_version() >= 1
    assert lib.spec_status_string(0) == b"ok"
    assert b"invalid" in lib.spec_status_string(1)


def test_workspace_bytes(spec):
    lib = spec.load()
    units = (151936 + 2047) // 2048
    n = lib.spec_workspace_bytes(128, 2048, 7, 151936)
    assert n >= 8 * units * (2048 + 128 * 7) + 8 * 2048
    assert lib.spec_workspace_bytes(-1, 1, 1, 1) == 0
    assert lib.spec_workspace_bytes(1, 1, 1, 0) == 0
    assert lib.spec_workspace_bytes(1, 1, 99, 10) == 0
    assert lib.spec_workspace_bytes(1, 1, 1, 524288) > 0  # SPEC_MAX_VOCAB
    assert lib.spec_workspace_bytes(1, 1, 1, 524289) == 0


def test_estimator_table_bytes(spec):
    lib = spec.load()
    e = spec.make_estimator({"beta": [0.0] * 15, "m_cap": 256})
    assert lib.spec_estimator_table_bytes(C.byref(e), 15) == 4 * (15 * 33 * 2 + 15 * 2 * 257)
    assert lib.spec_estimator_table_bytes(C.byref(e), 0) == 0
    e2 = spec.make_estimator({"constant_h": 0.9})
    assert lib.spec_estimator_table_bytes(C.byref(e2), 15) == 4


def _ws(spec):
    w = spec.WorkspaceStruct()
    w.base = 256 * 1024  # a fake, aligned device address; never dereferenced on these paths
    w.max_batch, w.max_rows, w.K, w.vocab = 4, 64, 7, 1024
    w.off_keys = 256  # the pricing keys' region, inside the stated size
    w.bytes = 256 + 4 * 1024 * 31
    return w


def test_host_validation_rejects_bad_arguments_without_a_gpu(spec):
    lib = spec.load()
    w = _ws(spec)
    P = 4096  # fake pointer, never dereferenced
    INV, UNS, WSE = 1, 3, 4
    # n-gram: n_min < 1, n_max < n_min, copy_cap < n_max, L beyond the limit
    args = lambda n_min, n_max, L, cap: (P, 64, P, 4, n_min, n_max, L, cap, P, P, P, P, P, C.byref(w), None)
    assert lib.spec_ngram_propose(*args(0, 3, 15, 256)) == INV
    assert lib.spec_ngram_propose(*args(4, 3, 15, 256)) == INV
    assert lib.spec_ngram_propose(*args(1, 15, 15, 10)) == INV
    assert lib.spec_ngram_propose(*args(1, 3, 32, 256)) == UNS
    assert lib.spec_ngram_propose(*args(1, 40, 15, 256)) == UNS
    # null pointer
    assert lib.spec_ngram_propose(P, 64, None, 4, 1, 3, 15, 256, P, P, P, P, P, C.byref(w), None) == INV
    # misaligned workspace; one too small for the pricing keys
    w2 = _ws(spec)
    w2.base = 256 * 1024 + 8
    assert lib.spec_ngram_propose(*args(1, 3, 15, 256)[:-2], C.byref(w2), None) == WSE
    w3 = _ws(spec)
    w3.bytes = 1024
    assert lib.spec_ngram_propose(*args(1, 3, 15, 256)[:-2], C.byref(w3), None) == WSE
    # pricing: K > L, negative budget, bad policy, oversized batch
    e = spec.make_estimator({"beta": [0.0] * 15})
    def price(B=4, K=7, L=15, budget=8, policy=0, lam=0.1, tb=1 << 20):
        return lib.spec_price_and_allocate(B, K, L, P, P, P, P, P, P, P, P, C.byref(e), P, tb, lam, budget, 15,
                                           policy, 1, P, P, P, P, P, P, P, C.byref(w), None)
    assert price(K=16, L=15) == INV
    assert price(budget=-1) == INV
    assert price(policy=9) == INV
    assert price(lam=float("nan")) == INV
    assert price(B=5000) == UNS
    assert price(L=40, K=7) == UNS
    assert price(tb=100) == INV  # a table too small for L
    # tree builder: Kc 0, width 0, too many candidates, too wide
    def tree(B=4, P=8, Kc=4, Lg=15, width=16, nc=1):
        return lib.spec_build_tree(B, P, Kc, P_, P_, P_, P_, nc, Lg, P_, P_, P_, width, P_, P_, P_, P_, C.byref(w),
                                   None)
    P_ = P
    assert tree(Kc=0) == INV
    assert tree(width=0) == INV
    assert tree(nc=0) == INV and tree(nc=10) == INV  # 1 <= n_chains <= P + 1
    assert tree(P=70, Kc=8) == UNS  # 1 + 560 + 15 candidates
    assert tree(nc=9, Lg=60) == UNS  # 1 + 32 + 540 candidates
    assert tree(width=257) == UNS
    assert lib.spec_build_tree(4, 8, 4, None, P, P, P, 1, 15, P, P, P, 16, P, P, P, P, C.byref(w), None) == INV
    # n-gram fill: n_min 0, copy_cap below n_min, negative depth, P + Lg too large, missing outputs
    def fill(B=4, stride=64, npos=8, Kc=4, n_min=4, cap=256, depth=32, Lg=32, tok=P):
        return lib.spec_ngram_fill(P, stride, P, B, npos, Kc, P, n_min, cap, depth, Lg, tok, P, P, C.byref(w), None)
    assert fill(n_min=0) == INV
    assert fill(n_min=5, cap=4) == INV
    assert fill(depth=-1) == INV
    assert fill(Kc=0) == INV
    assert fill(npos=4000, Lg=200) == UNS
    assert fill(tok=None) == INV
    assert fill(B=0, tok=None) == 0  # nothing to do: no device work
    # verification: vocab 0, bad dtype, batch beyond the workspace, NaN temperature
    def chain(B=4, V=1024, dtype=1, max_rows=64, T=0.0, K=0, draft=None):
        return lib.spec_verify_chain(B, V, dtype, P, P, max_rows, draft, K, P, 15, P, None, T, 0, 0, P, P, P,
                                     None, None, None, C.byref(w), None)
    assert chain(V=0) == INV
    assert chain(dtype=7) == INV
    assert chain(B=8) == WSE
    assert chain(max_rows=65) == WSE
    assert chain(V=2048) == WSE
    assert chain(T=float("nan")) == INV
    assert chain(draft=P, K=0) == INV
    # drafted verification: draft rows, point-mass flags and T > 0 required
    def drafted(T=1.0, draft=P, pm=P, K=7):
        return lib.spec_verify_chain_drafted(4, 1024, 1, P, P, 64, draft, K, P, 15, P, pm, T, 0, 0, P, P, P,
                                             None, None, None, C.byref(w), None)
    assert drafted(draft=None, K=0) == INV
    assert drafted(pm=None) == INV
    assert drafted(T=0.0) == INV
    # tree: too many nodes
    assert lib.spec_verify_tree(4, 1024, 1, P, P, 64, P, P, 300, P, P, P, C.byref(w), None) == UNS
    assert lib.spec_verify_tree(4, 1024, 1, P, None, 64, P, P, 16, P, P, P, C.byref(w), None) == INV
    # zero-sized batches are accepted without work
    assert lib.spec_verify_tree(0, 1024, 1, None, P, 0, None, None, 16, None, None, None, C.byref(w), None) == 0


def test_product_fails_loudly_without_the_library(spec, tmp_path):
    with pytest.raises(RuntimeError):
        spec.load(str(tmp_path / "missing.so"))
