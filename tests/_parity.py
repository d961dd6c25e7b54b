"""Helpers for GPU-vs-oracle parity tests (not collected by pytest).

The compare functions return a Parity record of what they compared and
append it to REPORT; tests/conftest.py prints REPORT at the end of the
session, so near-tie exclusions are counted and reported, never silent."""

from __future__ import annotations

import dataclasses
import math
import os

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


# band (in u units) around a CDF boundary inside which a float32 draw may land
# on the neighbouring token
CDF_BAND = 1e-5


def draw_in_band(weights, u, y):
    """True iff token y is the inverse-CDF draw of `weights` for some uniform
    within CDF_BAND of u (the oracle's exact draw is the case u itself)."""
    w = np.asarray(weights, dtype=np.float64)
    if y < 0 or y >= w.size or w[y] <= 0:
        return False
    c = np.cumsum(w)
    z = c[-1]
    lo = c[y - 1] / z if y > 0 else 0.0
    hi = c[y] / z
    return lo - CDF_BAND <= u <= hi + CDF_BAND


@dataclasses.dataclass
class Parity:
    """Outcome of one GPU-vs-oracle comparison over `sequences` sequences:
    `compared` were checked element by element, `near_tie_excluded` were
    left out because an accept test on the path lies within 1e-5 of its
    threshold (or a top-p cut sits at a near tie), and `cdf_band` of the
    compared ones drew a final token that is the float32 neighbour of the
    oracle's draw inside the CDF band.  `exact` = compared - cdf_band."""
    test: str
    sequences: int
    compared: int
    near_tie_excluded: int
    cdf_band: int

    @property
    def exact(self):
        return self.compared - self.cdf_band

    def as_dict(self):
        d = dataclasses.asdict(self)
        d["exact"] = self.exact
        return d


REPORT: list = []


def _record(seqs, compared, excluded, band, max_excluded):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    n = len(seqs)
    p = Parity(test, n, compared, excluded, band)
    REPORT.append(p)
    # a comparison must compare something, and exclusions stay under the
    # bound (default: a tenth of the sequences, at least one)
    bound = max(1, math.ceil(n / 10)) if max_excluded is None else max_excluded
    assert compared >= 1, p
    assert excluded <= bound, (p, bound)
    return p


def _check_final(ref, i, got, want):
    """Final (replacement / bonus) token: equal, or a float32 neighbour of a
    boundary draw.  Returns 1 if the band was needed."""
    if got == want:
        return 0
    w, u = ref.final[i]
    assert ref.sample_near is not None and ref.sample_near[i], (i, got, want)
    assert draw_in_band(w, u, got), (i, got, want, u)
    return 1


def compare_chain(gpu, ref, *, greedy=False, check_mass=True, seqs=None,
                  max_excluded=None):
    """gpu = (accepted, tokens, mass) tensors; ref = oracle ChainResult.
    Returns the Parity record (sequences compared, excluded as near ties --
    an accept test on the path within 1e-5 of its threshold, or a top-p cut
    -- and final draws inside the CDF band); asserts that at least one
    sequence was compared and that exclusions stay under `max_excluded`."""
    acc, tok, mass = (x.cpu().numpy() for x in gpu)
    B = ref.accepted.shape[0]
    seqs = list(range(B) if seqs is None else seqs)
    excluded = band = 0
    for i, b in enumerate(seqs):
        if ref.near_tie[i]:
            excluded += 1
            continue
        n = ref.accepted[i]
        assert acc[b] == n, (b, acc[b], n)
        assert np.array_equal(tok[b, :n], ref.tokens[i, :n]), b
        assert np.array_equal(tok[b, n + 1:], ref.tokens[i, n + 1:]), b
        if greedy:
            assert tok[b, n] == ref.tokens[i, n], b
        else:
            band += _check_final(ref, i, int(tok[b, n]), int(ref.tokens[i, n]))
    if check_mass:
        m = mass[seqs]
        if greedy:
            assert np.array_equal(m, ref.mass.astype(np.float32))
        else:
            np.testing.assert_allclose(m, ref.mass, rtol=MASS_RTOL,
                                       atol=MASS_ATOL)
    return _record(seqs, len(seqs) - excluded, excluded, band, max_excluded)


def compare_tree(gpu, ref, *, greedy=False, seqs=None, max_excluded=None,
                 mass_slack=None):
    """gpu = (path_len, path_nodes, tokens, mass); ref = oracle TreeResult.
    Returns the Parity record, with the same assertions as compare_chain.
    mass_slack ([len(seqs), N+1], optional): an absolute allowance added to
    the mass tolerance (the LM-head path's bound for logit roundings)."""
    plen, pnodes, tok, mass = (x.cpu().numpy() for x in gpu)
    B = ref.path_len.shape[0]
    seqs = list(range(B) if seqs is None else seqs)
    excluded = band = 0
    for i, b in enumerate(seqs):
        if ref.near_tie[i]:
            excluded += 1
            continue
        n = ref.path_len[i]
        assert plen[b] == n, (b, plen[b], n)
        assert np.array_equal(pnodes[b], ref.path_nodes[i]), b
        assert np.array_equal(tok[b, :n], ref.tokens[i, :n]), b
        assert np.array_equal(tok[b, n + 1:], ref.tokens[i, n + 1:]), b
        if greedy:
            assert tok[b, n] == ref.tokens[i, n], b
        else:
            band += _check_final(ref, i, int(tok[b, n]), int(ref.tokens[i, n]))
    m = mass[seqs]
    nan_g, nan_r = np.isnan(m), np.isnan(ref.mass)
    assert np.array_equal(nan_g, nan_r)
    if greedy:
        assert np.array_equal(m[~nan_g], ref.mass[~nan_r].astype(np.float32))
    elif mass_slack is None:
        np.testing.assert_allclose(m[~nan_g], ref.mass[~nan_r],
                                   rtol=MASS_RTOL, atol=MASS_ATOL)
    else:
        tol = MASS_RTOL * np.abs(ref.mass) + MASS_ATOL + mass_slack
        diff = np.abs(m - ref.mass)
        assert not (diff[~nan_r] > tol[~nan_r]).any(), float(
            (diff[~nan_r] / tol[~nan_r]).max())
    return _record(seqs, len(seqs) - excluded, excluded, band, max_excluded)
