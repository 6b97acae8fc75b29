"""The C-ABI library builds, loads, exports every symbol include/*.h declares,
and rejects bad arguments on the host before touching the GPU (no GPU is
needed: every call here fails validation before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from draft_lm_head_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(lmhead_\w+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lmhead_lowrank_score_topk", "lmhead_gather_logits", "lmhead_candidate_softmax",
                 "lmhead_two_stage", "lmhead_dense_head", "lmhead_pruned_head"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from draft_lm_head_gb300 import _lib
    names = declared_functions()
    assert names, "no declarations found"
    for name in names:
        assert hasattr(lib, name), f"{name} not exported"
    assert names == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_status_strings_and_version(lib):
    assert lib.lmhead_version() >= 100
    for st in range(0, -9, -1):
        assert lib.lmhead_status_string(st)
    assert lib.lmhead_status_string(-7).decode().startswith("device-side")


@pytest.mark.parametrize("mode,n,C,k,want", [
    (0, 4096, 128, 0, 128), (1, 4096, 128, 4, 128), (1, 128256, 256, 2, 1002),
    (1, 201088, 256, 2, 1572), (1, 151936, 256, 4, 2376), (1, 10, 4, 3, 8), (1, 10, 4, 2, 6),
    (0, 10, 11, 0, -2), (1, 10, 4, 5, -2), (1, 10, 0, 0, -2), (2, 10, 4, 1, -2), (0, 0, 1, 0, -2),
])
def test_candidate_count(lib, mode, n, C, k, want):
    assert lib.lmhead_candidate_count(mode, n, C, k) == want


def test_workspace_size(lib):
    loc = lib.lmhead_workspace_size(1, 128256, 4096, 256, 64, 256, 2)
    glo = lib.lmhead_workspace_size(0, 128256, 4096, 256, 64, 1024, 0)
    assert 0 < loc < glo and glo >= 64 * 128256 * 4
    assert lib.lmhead_workspace_size(1, 100, 12, 8, 1, 10, 1) == 0   # d not a multiple of 8
    assert lib.lmhead_workspace_size(0, 100, 16, 8, 1, 5000, 0) == 0  # C > n


def _p(v):
    return ctypes.c_void_p(v)


def test_validation_before_launch(lib):
    ok = 1 << 20  # a 16-byte aligned fake address; never dereferenced
    ws = 1 << 24
    big = 1 << 40
    args = lambda **kw: dict(dict(mode=1, W=ok, A=ok, B=ok, h=ok, tok=ok, n=1000, d=64, r=16, M=2,
                                  C=128, k=2, temp=1.0, ids=ok, lg=ok, q=ok, ws=ws, wsb=big), **kw)

    def call(a):
        return lib.lmhead_two_stage(a["mode"], _p(a["W"]), _p(a["A"]), _p(a["B"]), _p(a["h"]),
                                    _p(a["tok"]), a["n"], a["d"], a["r"], a["M"], a["C"], a["k"],
                                    a["temp"], _p(a["ids"]), _p(a["lg"]), _p(a["q"]), _p(a["ws"]),
                                    a["wsb"], None)

    assert call(args(W=None)) == -1
    assert call(args(q=None)) == -1
    assert call(args(d=60)) == -2
    assert call(args(r=12)) == -2
    assert call(args(M=0)) == -2
    assert call(args(k=200)) == -2
    assert call(args(C=0)) == -2
    assert call(args(mode=0, C=1001)) == -2
    assert call(args(mode=0, C=5000, n=10000)) == -5
    assert call(args(temp=0.0)) == -2
    assert call(args(temp=float("nan"))) == -2
    assert call(args(A=ok + 8)) == -3
    assert call(args(ws=ws + 16)) == -4
    assert call(args(ws=None)) == -4
    assert call(args(wsb=16)) == -4
    assert lib.lmhead_gather_logits(_p(ok), _p(ok), None, 100, 64, 1, 4, _p(ok), None) == -1
    assert lib.lmhead_gather_logits(_p(ok), _p(ok), _p(ok), 100, 63, 1, 4, _p(ok), None) == -2
    assert lib.lmhead_candidate_softmax(_p(ok), 1, 4, -1.0, _p(ok), None) == -2
    assert lib.lmhead_dense_head(_p(ok), _p(ok), 0, 64, 1, 1.0, _p(ok), None, None) == -2
    assert lib.lmhead_project_u(_p(ok), _p(ok + 4), 64, 16, 1, _p(ok), None) == -3


def test_speculative_entry_points_validate_before_launch(lib):
    ok = 1 << 20  # never dereferenced: validation returns first
    P = _p(ok)
    # draft selection: k_sel must be in [1, min(K, 16)]
    assert lib.lmhead_draft_select(None, P, 1, 8, 2, None, None, P, P, None, None, None, None) == -1
    assert lib.lmhead_draft_select(P, P, 1, 8, 0, None, None, P, P, None, None, None, None) == -2
    assert lib.lmhead_draft_select(P, P, 1, 8, 9, None, None, P, P, None, None, None, None) == -2
    assert lib.lmhead_draft_select(P, P, 1, 64, 17, None, None, P, P, None, None, None, None) == -2
    assert lib.lmhead_draft_select(P, P, 0, 8, 2, None, None, P, P, None, None, None, None) == -2
    assert lib.lmhead_draft_select(P, P, 1, 5000, 2, None, None, P, P, None, None, None, None) == -2
    # chain verification
    assert lib.lmhead_verify_chain(None, 100, 1, 2, P, P, P, 8, P, P, P, P, None) == -1
    assert lib.lmhead_verify_chain(P, 100, 1, 2, None, P, P, 8, P, P, P, P, None) == -1
    assert lib.lmhead_verify_chain(P, 0, 1, 2, P, P, P, 8, P, P, P, P, None) == -2
    assert lib.lmhead_verify_chain(P, 100, 1, -1, P, P, P, 8, P, P, P, P, None) == -2
    assert lib.lmhead_verify_chain(P, 100, 1, 2, P, P, P, 5000, P, P, P, P, None) == -2


def test_cluster_entry_points_validate_before_launch(lib):
    ok = 1 << 20  # never dereferenced: validation returns first
    P = _p(ok)
    assert lib.lmhead_cluster_candidate_count(128256, 128, 8) == 1024
    assert lib.lmhead_cluster_candidate_count(128256, 128, 1002) == 128256
    assert lib.lmhead_cluster_candidate_count(128256, 128, 1003) == -2  # more groups than exist
    assert lib.lmhead_cluster_candidate_count(1000, 128, 2) == -2  # ragged last group
    assert lib.lmhead_cluster_candidate_count(1024, 0, 2) == -2
    assert lib.lmhead_cluster_candidate_count(1024, 128, 0) == -2
    assert lib.lmhead_cluster_workspace_size(128256, 4096, 256, 64, 128, 8) > 64 * 1002 * 8
    assert lib.lmhead_cluster_workspace_size(1000, 4096, 256, 64, 128, 8) == 0

    def call(W=P, n=4096, d=256, r=32, M=1, group=128, G=4, T=1.0, groups=P, ws=P, wsb=1 << 30):
        return lib.lmhead_cluster_two_stage(W, P, P, P, n, d, r, M, group, G, T, groups, None, P,
                                            P, P, ws, wsb, None)

    assert call(W=None) == -1
    assert call(groups=None) == -1
    assert call(n=4000) == -2  # 128 does not divide n
    assert call(G=33) == -2
    assert call(d=100) == -2
    assert call(T=0.0) == -2
    assert call(n=1 << 20, group=128, G=4097) == -5  # past the group selector's budget
    assert call(W=_p(ok + 8)) == -3
    assert call(ws=None) == -4
    assert call(wsb=16) == -4


def _declarations():
    """name -> (return type text, [parameter type texts]) from include/*.h."""
    out = {}
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"([\w\s\*]+?)\b(lmhead_\w+)\s*\(([^;]*?)\)\s*;", text):
            ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
            plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
            out[name] = (ret.split()[-1] if ret else "", plist)
    return out


def _ctype_of(decl: str):
    c = ctypes
    if "*" in decl or decl.startswith("lmhead_stream"):
        return c.c_void_p
    if decl.startswith("int64_t"):
        return c.c_int64
    if decl.startswith("size_t"):
        return c.c_size_t
    if decl.startswith("float"):
        return c.c_float
    if decl.split()[0] in ("int", "int32_t"):
        return c.c_int
    raise AssertionError(f"unclassified parameter type: {decl}")


def test_binding_argument_types_match_the_header():
    """Every ctypes signature in the binding passes exactly the header's
    parameters, in order and by ABI class (pointer, int, int64, size_t,
    float): a mismatch would hand the library shifted arguments."""
    from draft_lm_head_gb300 import _lib
    decls = _declarations()
    assert set(decls) == set(_lib.SIGNATURES)
    for name, (ret, params) in decls.items():
        restype, argtypes = _lib.SIGNATURES[name]
        want = [_ctype_of(p) for p in params]
        assert list(argtypes) == want, name
        if ret.endswith("*") or ret == "char*":
            assert restype in (ctypes.c_char_p, ctypes.c_void_p), name
        else:
            assert restype == {"int": ctypes.c_int, "int64_t": ctypes.c_int64,
                               "size_t": ctypes.c_size_t}[ret], name
