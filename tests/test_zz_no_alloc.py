"""spec_verify_chain_noalloc: the chain verifier for callers that cannot
allocate device memory (an engine plugin given only its input and output
buffers, or a decode loop where cudaMalloc is not allowed).  Its scratch is a
fixed array inside the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row and checks each call's
outputs against spec_verify_chain on the same inputs, with the tolerance of
the other parity tests (integers exact, acceptance mass rel 1e-4).  This file
is collected last so that a run stopping at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

from tests._parity import MASS_ATOL, MASS_RTOL


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib
    _lib.load()
    return _lib


def _noalloc(lib, target, draft, toks, prm, out, stream):
    from speculative_decoding_verification_tree_gb300.api import _dt, _ptr
    B, K1, V = target.shape
    return lib.raw("spec_verify_chain_noalloc", _ptr(target), _ptr(draft),
                   _ptr(toks), B, K1 - 1, V, _dt(target), _dt(draft),
                   ctypes.byref(prm), _ptr(out[0]), _ptr(out[1]),
                   _ptr(out[2]), stream)


def test_noalloc_rejects_oversize_requests(lib):
    fake = ctypes.c_void_p(0x7f0000000000)  # never dereferenced
    prm = lib.SpecParams(1.0, 0, 1.0, 0, 0, 0, 0)
    rows_over = lib.SPEC_NOALLOC_MAX_ROWS // 5 + 1   # B*(K+1) too many rows
    assert lib.raw("spec_verify_chain_noalloc", fake, fake, fake, rows_over,
                   4, 1000, 0, 0, ctypes.byref(prm), fake, fake, fake,
                   None) == lib.SPEC_ERR_SHAPE
    # rows fit, argmax partials (rows * ceil(V / 16384)) do not
    assert lib.raw("spec_verify_chain_noalloc", fake, fake, fake, 1000, 4,
                   16384 * 14, 1, 1, ctypes.byref(prm), fake, fake, fake,
                   None) == lib.SPEC_ERR_SHAPE
    # sampling with top-k / top-p truncation needs candidate lists the
    # fixed array does not hold
    for top_k, top_p in ((50, 1.0), (0, 0.9), (50, 0.9)):
        tprm = lib.SpecParams(0.7, top_k, top_p, 0, 0, 0, 0)
        assert lib.raw("spec_verify_chain_noalloc", fake, fake, fake, 4, 4,
                       32000, 1, 1, ctypes.byref(tprm), fake, fake, fake,
                       None) == lib.SPEC_ERR_UNSUPPORTED
    # unaligned float32 rows too long for one cluster's shared memory: the
    # same SPEC_ERR_UNSUPPORTED as the workspace entry point, before any
    # GPU work
    assert lib.raw("spec_verify_chain_noalloc", fake, fake, fake, 1, 4,
                   300001, 0, 0, ctypes.byref(prm), fake, fake, fake,
                   None) == lib.SPEC_ERR_UNSUPPORTED
    # given draft normalisers are refused
    lprm = lib.SpecParams(1.0, 0, 1.0, 0, 0, 0, 0, 0x7f0000001000)
    assert lib.raw("spec_verify_chain_noalloc", fake, fake, fake, 4, 4,
                   32000, 1, 1, ctypes.byref(lprm), fake, fake, fake,
                   None) == lib.SPEC_ERR_ARG
    assert lib.raw("spec_get_status_noalloc", None, None) == lib.SPEC_ERR_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["sampled", "greedy"])
def test_noalloc_matches_workspace_entry_point_twice(lib, kind):
    import torch

    import synth
    from speculative_decoding_verification_tree_gb300 import api
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((21, 22)):  # two calls in a row
        if kind == "sampled":
            w = synth.workload("chain_sample", B=12, K=4, V=32000,
                               target_dtype=torch.bfloat16,
                               draft_dtype=torch.float32, seed=seed)
        else:
            w = synth.workload("greedy", B=64, K=8, V=128256, seed=seed)
        target, draft, toks = synth.chain_inputs(w, dev)
        B, K = toks.shape
        ws = api.workspace(lib.SPEC_OP_CHAIN, B, K, w.V, dev)
        want = api.spec_verify_chain(target, draft, toks,
                                     temperature=w.temperature,
                                     seed=w.decision_seed + call, ws=ws)
        out = (torch.full((B,), -7, dtype=torch.int32, device=dev),
               torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
               torch.full((B, K), -7.0, dtype=torch.float32, device=dev))
        prm = api.params(w.temperature, seed=w.decision_seed + call)
        rc = _noalloc(lib, target, draft, toks, prm, out, stream)
        assert rc == lib.SPEC_OK, rc
        torch.cuda.synchronize()
        # the status words of both calls agree (and report nothing here)
        st = ctypes.c_uint32(0xFFFFFFFF)
        assert lib.raw("spec_get_status_noalloc", ctypes.byref(st),
                       stream) == lib.SPEC_OK
        assert st.value == api.spec_get_status(ws) == 0, st.value
        assert np.array_equal(out[0].cpu().numpy(), want[0].cpu().numpy())
        assert np.array_equal(out[1].cpu().numpy(), want[1].cpu().numpy())
        np.testing.assert_allclose(out[2].cpu().numpy(),
                                   want[2].cpu().numpy(), rtol=MASS_RTOL,
                                   atol=MASS_ATOL)
