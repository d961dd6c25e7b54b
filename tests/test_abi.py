"""Host-only checks of the C ABI: the library builds, loads and exports every
symbol include/specverify.h declares, and rejects bad arguments before any
device work (these calls never reach the GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib
    return _lib


def _declared():
    src = open(os.path.join(ROOT, "include", "specverify.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 8
    handle = lib.load()
    for n in names:
        assert hasattr(handle, n), n
    assert set(names) == set(lib.EXPORTED)


def test_params_struct_layout(lib):
    P = lib.SpecParams
    assert ctypes.sizeof(P) == 40
    assert P.seed.offset == 16 and P.philox_offset.offset == 24
    assert P.draft_lse.offset == 32


def test_workspace_sizes(lib):
    f = lib.load().spec_workspace_bytes
    assert f(lib.SPEC_OP_CHAIN, 4, 5, 1000) % 256 == 0
    assert f(lib.SPEC_OP_CHAIN, 4, 5, 1000) > 0
    assert f(lib.SPEC_OP_TREE, 0, 0, 1) > 0
    assert f(lib.SPEC_OP_CHAIN, -1, 5, 1000) == 0
    assert f(lib.SPEC_OP_TREE, 1, 5000, 1000) == 0
    assert f(lib.SPEC_OP_CHAIN, 1, 5, 0) == 0
    assert f(99, 1, 5, 10) == 0
    assert f(lib.SPEC_OP_EAGLE2, 128, 51, 128256) > 128 * 51 * 8


def _prm(lib, **kw):
    d = dict(temperature=1.0, top_k=0, top_p=1.0, draft_kind=0, seed=0,
             philox_offset=0, flags=0)
    d.update(kw)
    return lib.SpecParams(**d)


FAKE = ctypes.c_void_p(0x7f0000000000)  # never dereferenced: calls fail early


def _chain(lib, B=2, K=3, V=100, prm=None, ws=FAKE, ws_bytes=1 << 20,
           target=FAKE, draft=FAKE, dt=0):
    prm = prm or _prm(lib)
    return lib.raw("spec_verify_chain", target, draft, FAKE, B, K, V, dt, dt,
                   ctypes.byref(prm), FAKE, FAKE, FAKE, ws, ws_bytes, None)


def test_chain_argument_errors(lib):
    assert _chain(lib, B=-1) == lib.SPEC_ERR_SHAPE
    assert _chain(lib, V=0) == lib.SPEC_ERR_SHAPE
    assert _chain(lib, K=5000) == lib.SPEC_ERR_SHAPE
    assert _chain(lib, dt=7) == lib.SPEC_ERR_DTYPE
    assert _chain(lib, target=None) == lib.SPEC_ERR_ARG
    assert _chain(lib, draft=None) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, temperature=-1.0)) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, temperature=float("nan"))) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, top_p=0.0)) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, top_p=1.5)) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, top_k=-2)) == lib.SPEC_ERR_ARG
    assert _chain(lib, prm=_prm(lib, draft_kind=3)) == lib.SPEC_ERR_DTYPE
    assert _chain(lib, prm=_prm(lib, flags=1)) == lib.SPEC_ERR_ARG
    # given draft normalisers are a tree-verification input only
    assert _chain(lib, prm=_prm(lib, draft_lse=FAKE.value)) == lib.SPEC_ERR_ARG
    # top-p alone keeps up to V tokens: fine for V <= 128, not beyond
    assert _chain(lib, V=1000, prm=_prm(lib, top_p=0.9)) == \
        lib.SPEC_ERR_UNSUPPORTED
    assert _chain(lib, V=5000, prm=_prm(lib, top_k=2000)) == \
        lib.SPEC_ERR_UNSUPPORTED
    # an odd row length too long for the general kernel's shared memory
    big = lib.raw("spec_workspace_bytes", lib.SPEC_OP_CHAIN, 2, 3, 700001)
    assert _chain(lib, V=700001, ws_bytes=big) == lib.SPEC_ERR_UNSUPPORTED
    assert _chain(lib, ws=None) == lib.SPEC_ERR_WORKSPACE
    assert _chain(lib, ws=ctypes.c_void_p(0x7f0000000010)) == \
        lib.SPEC_ERR_WORKSPACE
    assert _chain(lib, ws_bytes=16) == lib.SPEC_ERR_WORKSPACE
    # greedy needs no draft
    assert _chain(lib, draft=None, ws=None,
                  prm=_prm(lib, temperature=0.0)) == lib.SPEC_ERR_WORKSPACE


def test_tree_and_mask_argument_errors(lib):
    prm = _prm(lib)
    f = lib.raw
    assert f("spec_verify_tree", FAKE, FAKE, FAKE, FAKE, FAKE, 1, -1, 1, 10,
             0, 0, ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20,
             None) == lib.SPEC_ERR_SHAPE
    assert f("spec_verify_tree", FAKE, FAKE, None, FAKE, FAKE, 1, 3, 4, 10,
             0, 0, ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20,
             None) == lib.SPEC_ERR_ARG
    # given draft normalisers: logit drafts without truncation only
    for kw in (dict(draft_kind=1), dict(top_k=5), dict(top_p=0.5)):
        p = _prm(lib, draft_lse=FAKE.value, **kw)
        assert f("spec_verify_tree", FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 4,
                 100, 0, 0, ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE,
                 1 << 20, None) == lib.SPEC_ERR_ARG, kw
    assert f("spec_tree_mask", FAKE, 1, 65, None, FAKE, None) == \
        lib.SPEC_ERR_SHAPE
    assert f("spec_tree_mask", FAKE, 1, 5, None, None, None) == \
        lib.SPEC_ERR_ARG
    assert f("spec_tree_mask", FAKE, -1, 5, FAKE, None, None) == \
        lib.SPEC_ERR_SHAPE


def test_eagle2_argument_errors(lib):
    prm = _prm(lib, temperature=0.8)
    f = lib.raw

    def call(B=2, V=1000, dt=1, depth=6, topk=10, width=10, total=60,
             p=prm, ws_bytes=1 << 24):
        return f("spec_eagle2_expand_rerank", FAKE, B, V, dt, depth, topk,
                 width, total, ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE,
                 FAKE, ws_bytes, None)
    assert call(topk=40) == lib.SPEC_ERR_SHAPE
    assert call(topk=11, V=10) == lib.SPEC_ERR_SHAPE
    assert call(total=511) == lib.SPEC_ERR_SHAPE
    assert call(depth=0) == lib.SPEC_ERR_SHAPE
    assert call(dt=4) == lib.SPEC_ERR_DTYPE
    assert call(p=_prm(lib, temperature=0.0)) == lib.SPEC_ERR_ARG
    assert call(ws_bytes=8) == lib.SPEC_ERR_WORKSPACE


def test_kv_commit_argument_errors(lib):
    f = lib.raw

    def call(B=2, n1=1, n2=1, sb=256, s1=0, s2=0, sp=16, row=16, kv=FAKE,
             pre=FAKE, nodes=FAKE, plen=FAKE, N=4, out=FAKE):
        return f("spec_kv_commit", kv, B, n1, n2, sb, s1, s2, sp, row, pre,
                 nodes, plen, N, out, None)
    assert call(B=-1) == lib.SPEC_ERR_SHAPE
    assert call(N=-1) == lib.SPEC_ERR_SHAPE
    assert call(row=-16) == lib.SPEC_ERR_SHAPE
    assert call(sp=-16) == lib.SPEC_ERR_SHAPE
    assert call(pre=None) == lib.SPEC_ERR_ARG
    assert call(plen=None) == lib.SPEC_ERR_ARG
    assert call(out=None) == lib.SPEC_ERR_ARG
    assert call(kv=None) == lib.SPEC_ERR_ARG          # a tree moves entries
    assert call(B=0, kv=None, pre=None, plen=None, out=None) == lib.SPEC_OK


def test_error_strings(lib):
    h = lib.load()
    for code in range(-6, 1):
        assert h.spec_error_string(code)
    assert h.spec_error_string(-99) == b"unknown error"


def test_accept_stats_argument_errors(lib):
    f = lib.raw
    rec = lib.SpecAcceptStats()
    assert ctypes.sizeof(rec) == 9 * 8

    def call(count=FAKE, parent=FAKE, path=FAKE, conf=FAKE, B=2, n=4,
             nbins=10, out=ctypes.byref(rec)):
        return f("spec_accept_stats", count, parent, path, conf, B, n, nbins,
                 out, None)
    assert call(count=None) == lib.SPEC_ERR_ARG
    assert call(out=None) == lib.SPEC_ERR_ARG
    assert call(parent=None) == lib.SPEC_ERR_ARG      # one of the pair
    assert call(path=None) == lib.SPEC_ERR_ARG
    assert call(B=-1) == lib.SPEC_ERR_SHAPE
    assert call(n=0) == lib.SPEC_ERR_SHAPE
    assert call(n=1025) == lib.SPEC_ERR_SHAPE
    assert call(nbins=0) == lib.SPEC_ERR_SHAPE
    assert call(nbins=lib.SPEC_STATS_MAX_BINS + 1) == lib.SPEC_ERR_SHAPE
    # without confidences the bin count is not used; B = 0 does nothing
    assert call(conf=None, nbins=0, B=0) == lib.SPEC_OK
    assert call(parent=None, path=None, B=0) == lib.SPEC_OK
    # misaligned arrays are argument errors, caught before any launch
    odd = ctypes.c_void_p(0x7f0000000002)
    assert call(count=odd) == lib.SPEC_ERR_ARG
    assert call(conf=odd) == lib.SPEC_ERR_ARG
    rec.len_hist = 0x7f0000000004
    assert call() == lib.SPEC_ERR_ARG
    rec.len_hist = None


def test_tree_attention_argument_errors(lib):
    f = lib.raw

    def call(B=2, N=8, Hq=8, Hkv=2, D=128, S=64, scale=0.1, q=FAKE, k=FAKE,
             v=FAKE, out=FAKE):
        return f("spec_tree_attention", q, k, v, FAKE, FAKE, B, N, Hq, Hkv, D,
                 S, ctypes.c_float(scale), out, None)
    assert call(N=0) == lib.SPEC_ERR_SHAPE
    assert call(N=65) == lib.SPEC_ERR_SHAPE
    assert call(Hq=6, Hkv=4) == lib.SPEC_ERR_SHAPE
    assert call(S=4) == lib.SPEC_ERR_SHAPE
    assert call(B=-1) == lib.SPEC_ERR_SHAPE
    assert call(B=65536) == lib.SPEC_ERR_SHAPE
    assert call(D=64) == lib.SPEC_ERR_UNSUPPORTED
    assert call(scale=0.0) == lib.SPEC_ERR_ARG
    assert call(scale=float("inf")) == lib.SPEC_ERR_ARG
    assert call(q=None) == lib.SPEC_ERR_ARG
    assert call(k=ctypes.c_void_p(0x7f0000000008)) == lib.SPEC_ERR_ARG
    assert f("spec_tree_attention", FAKE, FAKE, FAKE, FAKE,
             ctypes.c_void_p(0x7f0000000004), 2, 8, 8, 2, 128, 64,
             ctypes.c_float(0.1), FAKE, None) == lib.SPEC_ERR_ARG
    assert call(B=0, q=None, out=None) == lib.SPEC_OK


def test_lm_head_argument_errors(lib):
    f = lib.raw
    ws_ok = lib.raw("spec_workspace_bytes", lib.SPEC_OP_LMHEAD, 10, 0, 1000)
    assert ws_ok > 10 * 4 * 8 and ws_ok % 256 == 0
    assert f("spec_workspace_bytes", lib.SPEC_OP_LMHEAD, 10, 3, 1000) == 0
    t = lib.raw("spec_workspace_bytes", lib.SPEC_OP_TREE_LMHEAD, 2, 5, 1000)
    # the logits of every tree row are part of the workspace
    assert t > lib.raw("spec_workspace_bytes", lib.SPEC_OP_TREE, 2, 5,
                       1000) + 2 * 6 * 1000 * 2

    def lm(M=10, H=64, V=1000, T=1.0, hidden=FAKE, w=FAKE, out=FAKE,
           lse=None, ws=FAKE, nbytes=None):
        return f("spec_lm_head", hidden, w, M, H, V, ctypes.c_float(T), out,
                 lse, ws, ws_ok if nbytes is None else nbytes, None)
    assert lm(M=-1) == lib.SPEC_ERR_SHAPE
    assert lm(V=0) == lib.SPEC_ERR_SHAPE
    assert lm(H=0) == lib.SPEC_ERR_SHAPE
    assert lm(T=-1.0) == lib.SPEC_ERR_ARG
    assert lm(T=0.0, lse=FAKE) == lib.SPEC_ERR_ARG  # normalisers need T > 0
    assert lm(out=None) == lib.SPEC_ERR_ARG
    assert lm(H=60) == lib.SPEC_ERR_UNSUPPORTED       # rows not 16-byte multiples
    assert lm(w=ctypes.c_void_p(0x7f0000000008)) == lib.SPEC_ERR_UNSUPPORTED
    assert lm(nbytes=ws_ok - 1) == lib.SPEC_ERR_WORKSPACE
    assert lm(ws=ctypes.c_void_p(0x7f0000000010)) == lib.SPEC_ERR_WORKSPACE

    prm = _prm(lib)

    def tree(B=2, N=5, R=6, V=1000, H=64, hidden=FAKE, nbytes=None, p=prm):
        return f("spec_verify_tree_lmhead", hidden, FAKE, H, FAKE, FAKE, FAKE,
                 FAKE, B, N, R, V, 0, ctypes.byref(p), FAKE, FAKE, FAKE,
                 FAKE, None, FAKE, t if nbytes is None else nbytes, None)
    assert tree(B=-1) == lib.SPEC_ERR_SHAPE
    assert tree(N=5000) == lib.SPEC_ERR_SHAPE
    assert tree(H=12) == lib.SPEC_ERR_UNSUPPORTED
    assert tree(hidden=None) == lib.SPEC_ERR_ARG
    assert tree(nbytes=t - 256) == lib.SPEC_ERR_WORKSPACE
    assert tree(p=_prm(lib, flags=1)) == lib.SPEC_ERR_ARG
    # the test-only stall flag passes the parameter check here (the call
    # then stops at the short workspace) and nowhere else
    stall = _prm(lib, flags=lib.SPEC_FLAG_TEST_STALL)
    assert tree(p=stall, nbytes=t - 256) == lib.SPEC_ERR_WORKSPACE
    assert f("spec_verify_tree", FAKE, FAKE, FAKE, FAKE, FAKE, 2, 5, 6, 1000,
             1, 0, ctypes.byref(stall), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30,
             None) == lib.SPEC_ERR_ARG
    assert tree(p=_prm(lib, top_k=500)) == lib.SPEC_ERR_UNSUPPORTED


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_compiles_for_plain_c_and_cpp_callers(tmp_path, lang, std):
    # the boundary is a C ABI: the header must stand alone in C and C++
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "specverify.h"\n'
                   "int main(void) { spec_params_t p; spec_accept_stats_t r;\n"
                   "  (void)p; (void)r; return SPEC_OK; }\n")
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic",
                        "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-fsyntax-only", str(src)], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
