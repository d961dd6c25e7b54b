"""Host-side checks of the Python binding (no GPU, no library call): every
wrapper in api.py passes exactly the arguments its C signature declares, in
a form ctypes accepts, and rejects malformed tensors before any call."""

import ctypes

import pytest
import torch

from speculative_decoding_verification_tree_gb300 import _lib, api


@pytest.fixture
def captured(monkeypatch):
    calls = []

    def fake_call(name, *args):
        argtypes = _lib._SIGNATURES[name][1]
        assert len(args) == len(argtypes), (name, len(args), len(argtypes))
        for a, t in zip(args, argtypes):
            if a is None:
                continue
            if t is ctypes.c_void_p:
                assert isinstance(a, (ctypes.c_void_p, int)), (name, a)
            elif isinstance(t, type) and issubclass(t, ctypes._Pointer):
                assert isinstance(a, type(ctypes.byref(ctypes.c_int()))), (name, a)
            else:
                t(a)  # a value ctypes can convert
        calls.append((name, args))
        return 0

    monkeypatch.setattr(_lib, "call", fake_call)
    # device pointers are not needed: any tensor maps to a fake address
    monkeypatch.setattr(api, "_ptr", lambda t: None if t is None
                        else ctypes.c_void_p(0x7f0000000000))
    monkeypatch.setattr(api, "_stream", lambda s: ctypes.c_void_p(0))
    monkeypatch.setattr(api, "workspace", lambda op, B, n, V, device=None:
                        torch.empty(256, dtype=torch.uint8))
    return calls


def test_verify_wrappers_match_their_signatures(captured):
    B, K, V = 2, 3, 64
    t = torch.zeros(B, K + 1, V)
    d = torch.zeros(B, K, V)
    tok = torch.zeros(B, K, dtype=torch.int32)
    api.spec_verify_chain(t, d, tok, temperature=0.7, top_k=5)
    N = 4
    tt = torch.zeros(B, N + 1, V)
    dd = torch.zeros(B, N + 1, V)
    qr = torch.zeros(B, N + 1, dtype=torch.int32)
    nt = torch.zeros(B, N, dtype=torch.int32)
    par = torch.zeros(B, N, dtype=torch.int32)
    api.spec_verify_tree(tt, dd, qr, nt, par, temperature=1.0)
    api.spec_tree_mask(par, bits=True)
    api.spec_eagle2_expand_rerank(torch.zeros(B, 51, V, dtype=torch.bfloat16),
                                  temperature=0.8)
    H = 64
    api.spec_lm_head(torch.zeros(B, N + 1, H, dtype=torch.bfloat16),
                     torch.zeros(V, H, dtype=torch.bfloat16), temperature=1.0,
                     row_lse=True)
    api.spec_verify_tree_lmhead(torch.zeros(B, N + 1, H, dtype=torch.bfloat16),
                                torch.zeros(V, H, dtype=torch.bfloat16), dd,
                                qr, nt, par, temperature=1.0,
                                draft_kind="probs")
    assert [c[0] for c in captured] == ["spec_verify_chain", "spec_verify_tree",
                                        "spec_tree_mask",
                                        "spec_eagle2_expand_rerank",
                                        "spec_lm_head",
                                        "spec_verify_tree_lmhead"]


def test_post_verification_wrappers_match_their_signatures(captured):
    B, n = 3, 6
    api.spec_accept_stats(torch.zeros(B, dtype=torch.int32),
                          torch.zeros(B, n, dtype=torch.int32),
                          torch.zeros(B, n, dtype=torch.int32),
                          torch.zeros(B, n), n=n, nbins=8,
                          out={f: None for f in _lib.STATS_FIELDS})
    q = torch.zeros(B, n, 4, 128, dtype=torch.bfloat16)
    kv = torch.zeros(B, 2, 16, 128, dtype=torch.bfloat16)
    api.spec_tree_attention(q, kv, kv, torch.zeros(B, dtype=torch.int32),
                            torch.zeros(B, n, dtype=torch.int64), out=q)
    api.spec_kv_commit(torch.zeros(64, dtype=torch.uint8),
                       torch.zeros(B, dtype=torch.int32),
                       torch.zeros(B, dtype=torch.int32),
                       torch.zeros(B, n, dtype=torch.int32),
                       layout=(1, 1, 0, 0, 0, 16), row_bytes=16, N=n,
                       new_len=torch.zeros(B, dtype=torch.int32))
    names = [c[0] for c in captured]
    assert names == ["spec_accept_stats", "spec_tree_attention",
                     "spec_kv_commit"]
    # the records struct carries the nine record pointers in header order
    rec = captured[0][1][7]._obj
    assert isinstance(rec, _lib.SpecAcceptStats)
    assert [f for f, _ in rec._fields_] == list(_lib.STATS_FIELDS)


def test_wrappers_reject_malformed_tensors(captured):
    with pytest.raises(ValueError):
        api.spec_accept_stats(torch.zeros(3, dtype=torch.int64), n=4)
    with pytest.raises(ValueError):  # parent without path_nodes
        api.spec_accept_stats(torch.zeros(3, dtype=torch.int32),
                              torch.zeros(3, 4, dtype=torch.int32), n=4)
    with pytest.raises(ValueError):
        api.spec_accept_stats(torch.zeros(3, dtype=torch.int32), n=4,
                              confidence=torch.zeros(3, 5))
    q = torch.zeros(1, 2, 2, 128, dtype=torch.bfloat16)
    kv = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # 32-bit mask rows
        api.spec_tree_attention(q, kv, kv, torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, 2, dtype=torch.int32))
    with pytest.raises(ValueError):  # float32 queries
        api.spec_tree_attention(q.float(), kv, kv,
                                torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, 2, dtype=torch.int64))
    with pytest.raises(ValueError):  # 32-bit records would be overrun
        api.spec_accept_stats(torch.zeros(3, dtype=torch.int32), n=4,
                              out={"len_hist": torch.zeros(5,
                                                           dtype=torch.int32)})
    with pytest.raises(ValueError):  # records sized for another n
        api.spec_accept_stats(torch.zeros(3, dtype=torch.int32), n=4,
                              out={"node_tested": torch.zeros(
                                  5, dtype=torch.int64)})
    with pytest.raises(ValueError):  # output of the wrong shape
        api.spec_tree_attention(q, kv, kv, torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, 2, dtype=torch.int64),
                                out=torch.zeros(1, 2, 2, 64,
                                                dtype=torch.bfloat16))
    assert captured == []


def test_verification_wrappers_reject_wrong_outputs(captured):
    B, K, V = 2, 3, 64
    t, d = torch.zeros(B, K + 1, V), torch.zeros(B, K, V)
    tok = torch.zeros(B, K, dtype=torch.int32)
    bad = (torch.empty(B, dtype=torch.int64),          # accepted as int64
           torch.empty(B, K + 1, dtype=torch.int32),
           torch.empty(B, K))
    with pytest.raises(ValueError):
        api.spec_verify_chain(t, d, tok, out=bad)
    N = 5
    short = (torch.empty(B, dtype=torch.int32),
             torch.empty(B, N, dtype=torch.int32),
             torch.empty(B, N, dtype=torch.int32),      # one token short
             torch.empty(B, N + 1))
    with pytest.raises(ValueError):
        api.spec_verify_tree(torch.zeros(B, N + 1, V), torch.zeros(B, N + 1, V),
                             torch.zeros(B, N + 1, dtype=torch.int32),
                             torch.zeros(B, N, dtype=torch.int32),
                             torch.zeros(B, N, dtype=torch.int32), out=short)
    with pytest.raises(ValueError):
        api.spec_kv_commit(torch.zeros(8, dtype=torch.uint8),
                           torch.zeros(B, dtype=torch.int32),
                           torch.zeros(B, dtype=torch.int32), None,
                           layout=(1, 1, 0, 0, 0, 16), row_bytes=16, N=4,
                           new_len=torch.zeros(B, dtype=torch.int64))
    assert captured == []


def test_wrappers_reject_tensors_on_another_device(captured):
    """Every tensor of a call (inputs, outputs, workspace) must be on the
    primary input's device: the library launches on that device and would
    otherwise dereference another device's memory.  A tensor on the meta
    device stands in for one on another GPU."""
    B, K, V = 2, 3, 64
    t = torch.zeros(B, K + 1, V)
    d = torch.zeros(B, K, V)
    tok = torch.zeros(B, K, dtype=torch.int32)
    other = lambda *s, dtype=torch.float32: torch.empty(*s, dtype=dtype,
                                                        device="meta")
    with pytest.raises(ValueError, match="same|must be on"):
        api.spec_verify_chain(t, other(B, K, V), tok, temperature=1.0)
    with pytest.raises(ValueError, match="must be on"):
        api.spec_verify_chain(t, d, tok, temperature=1.0,
                              out=(other(B, dtype=torch.int32),
                                   torch.zeros(B, K + 1, dtype=torch.int32),
                                   torch.zeros(B, K)))
    with pytest.raises(ValueError, match="must be on"):
        api.spec_verify_chain(t, d, tok, temperature=1.0,
                              ws=other(256, dtype=torch.uint8))
    N = 4
    tt = torch.zeros(B, N + 1, V)
    qr = torch.zeros(B, N + 1, dtype=torch.int32)
    nt = torch.zeros(B, N, dtype=torch.int32)
    par = torch.zeros(B, N, dtype=torch.int32)
    with pytest.raises(ValueError, match="must be on"):
        api.spec_verify_tree(tt, tt, qr, nt, other(B, N, dtype=torch.int32),
                             temperature=1.0)
    q = torch.zeros(B, N, 4, 128, dtype=torch.bfloat16)
    kv = torch.zeros(B, 2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be on"):
        api.spec_tree_attention(q, kv, other(B, 2, 16, 128,
                                             dtype=torch.bfloat16),
                                torch.zeros(B, dtype=torch.int32),
                                torch.zeros(B, N, dtype=torch.int64))
    with pytest.raises(ValueError, match="must be on"):
        api.spec_accept_stats(torch.zeros(B, dtype=torch.int32), par,
                              other(B, N, dtype=torch.int32), n=N)
    with pytest.raises(ValueError, match="must be on"):
        api.spec_kv_commit(torch.zeros(64, dtype=torch.uint8),
                           torch.zeros(B, dtype=torch.int32),
                           other(B, dtype=torch.int32), None,
                           layout=(1, 1, 0, 0, 0, 16), row_bytes=16, N=N)
    assert captured == []  # nothing reached the library
