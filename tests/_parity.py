"""Helpers for GPU-vs-oracle parity tests (not collected by pytest)."""

from __future__ import annotations

import numpy as np
import torch

# float tolerance of the acceptance mass: float32 accumulation over bf16 /
# float32 logits against the float64 oracle
MASS_RTOL = 1e-4
MASS_ATOL = 1e-6


def lib_ready():
    """Build the library if needed and make sure a GPU is present."""
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_tree_gb300 import _lib
    _lib.load()


def np64(t):
    if t is None:
        return None
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare_chain(gpu, ref, *, greedy=False, check_mass=True, seqs=None):
    """gpu = (accepted, tokens, mass) tensors; ref = oracle ChainResult.
    Returns the number of sequences excluded as near ties."""
    acc, tok, mass = (x.cpu().numpy() for x in gpu)
    B = ref.accepted.shape[0]
    seqs = range(B) if seqs is None else seqs
    excluded = 0
    for i, b in enumerate(seqs):
        if ref.near_tie[i]:
            excluded += 1
            continue
        assert acc[b] == ref.accepted[i], (b, acc[b], ref.accepted[i])
        assert np.array_equal(tok[b], ref.tokens[i]), (b, tok[b], ref.tokens[i])
    if check_mass:
        m = mass[list(seqs)]
        if greedy:
            assert np.array_equal(m, ref.mass.astype(np.float32))
        else:
            np.testing.assert_allclose(m, ref.mass, rtol=MASS_RTOL,
                                       atol=MASS_ATOL)
    return excluded


def compare_tree(gpu, ref, *, greedy=False, seqs=None):
    plen, pnodes, tok, mass = (x.cpu().numpy() for x in gpu)
    B = ref.path_len.shape[0]
    seqs = range(B) if seqs is None else seqs
    excluded = 0
    for i, b in enumerate(seqs):
        if ref.near_tie[i]:
            excluded += 1
            continue
        assert plen[b] == ref.path_len[i], (b, plen[b], ref.path_len[i])
        assert np.array_equal(pnodes[b], ref.path_nodes[i]), b
        assert np.array_equal(tok[b], ref.tokens[i]), (b, tok[b], ref.tokens[i])
    m = mass[list(seqs)]
    nan_g, nan_r = np.isnan(m), np.isnan(ref.mass)
    assert np.array_equal(nan_g, nan_r)
    if greedy:
        assert np.array_equal(m[~nan_g], ref.mass[~nan_r].astype(np.float32))
    else:
        np.testing.assert_allclose(m[~nan_g], ref.mass[~nan_r],
                                   rtol=MASS_RTOL, atol=MASS_ATOL)
    return excluded
