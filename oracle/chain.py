"""Chain verification (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows the verify listing of "064 · 投机解码" (section 三) and steps 3-4 of the
draft/verify loop of "投机解码与 EAGLE" ("每步" list):

* for k = 0 .. K-1, left to right: accept drafted token x_k iff
  u(b, k, 0) < p_k(x_k) / q_k(x_k);
* at the first rejection, sample the replacement from norm(max(0, p_k - q_k))
  with u(b, k, 1) and stop;
* if every token is accepted, sample a bonus token from p_K with u(b, K, 1).

The acceptance mass alpha_k = sum_x min(p_k, q_k) is reported for every row
k < K, including rows after the first rejection.

Temperature 0 uses the greedy simplification of "投机解码与 EAGLE": accept
while x_k equals argmax of the target logits, then emit that argmax; alpha_k
is then the indicator 1[x_k == argmax].  No draft rows are read.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox
from .sampling import (accept, acceptance_mass, argmax_first, inverse_cdf,
                       residual, transform)

# Status bits (same meaning as the library's SPEC_STATUS_* flags).
ST_QZERO_ACCEPT = 2
ST_RESIDUAL_ZERO = 4
ST_DRAFT_EXHAUSTED = 8
ST_BAD_TREE = 32
ST_TOKEN_RANGE = 64


@dataclass
class ChainResult:
    accepted: np.ndarray      # [B] int32
    tokens: np.ndarray        # [B, K+1] int32, -1 padded
    mass: np.ndarray          # [B, K] float64
    near_tie: np.ndarray      # [B] bool: an accept test or a top-p cut on
                              # the path was within NEAR_TIE of its threshold
    status: int = 0
    near_rows: list = field(default_factory=list)  # (b, k) of near-tie rows
    sample_near: np.ndarray = None  # [B] bool: final draw near a CDF boundary
    final: list = field(default_factory=list)      # per b: (weights, u)


def verify_chain(target, draft, draft_tokens, *, temperature: float,
                 top_k: int = 0, top_p: float = 1.0, draft_kind="logits",
                 seed: int = 0, offset: int = 0, uniform=None,
                 batch_ids=None) -> ChainResult:
    """target [B, K+1, V], draft [B, K, V] (or None when temperature == 0),
    draft_tokens [B, K].  ``uniform(b, i, slot)`` overrides Philox."""
    target = np.asarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    toks = np.asarray(draft_tokens).reshape(B, K)
    if uniform is None:
        # batch_ids: the sequence index each row had in the full batch (the
        # Philox counter uses it), when the oracle checks a subset
        ids = list(range(B)) if batch_ids is None else [int(x) for x in
                                                         batch_ids]

        def uniform(b, i, slot):
            return philox.uniform(seed, ids[b], i, slot, offset)

    accepted = np.zeros(B, dtype=np.int32)
    out = np.full((B, K + 1), -1, dtype=np.int32)
    mass = np.zeros((B, K), dtype=np.float64)
    near = np.zeros(B, dtype=bool)
    status = 0
    near_rows = []

    snear = np.zeros(B, dtype=bool)
    final = []
    if temperature == 0:
        for b in range(B):
            g = [argmax_first(target[b, k]) for k in range(K + 1)]
            n = K
            for k in range(K):
                mass[b, k] = 1.0 if toks[b, k] == g[k] else 0.0
            for k in range(K):
                if toks[b, k] != g[k]:
                    n = k
                    break
            accepted[b] = n
            out[b, :n] = toks[b, :n]
            out[b, n] = g[n]
        return ChainResult(accepted, out, mass, near, status, near_rows,
                           snear, final)

    draft = np.asarray(draft)
    for b in range(B):
        ps, qs = [], []
        for k in range(K + 1):
            p, nt = transform(target[b, k], "logits", temperature, top_k, top_p)
            if nt:
                near_rows.append((b, k))
            ps.append(p)
        for k in range(K):
            q, nt = transform(draft[b, k], draft_kind, temperature, top_k,
                              top_p)
            if nt:
                near_rows.append((b, k))
            qs.append(q)
            mass[b, k] = acceptance_mass(ps[k], q)
        path_near = any(r[0] == b for r in near_rows)
        n = K
        for k in range(K):
            x = int(toks[b, k])
            if not 0 <= x < V:
                ok, nt, qz = False, False, False
                status |= ST_TOKEN_RANGE
            else:
                ok, nt, qz = accept(ps[k], qs[k], x, uniform(b, k, 0))
            path_near |= nt
            if qz:
                status |= ST_QZERO_ACCEPT
            if not ok:
                n = k
                break
        if n < K:
            w, fb = residual(ps[n], qs[n])
            if fb:
                status |= ST_RESIDUAL_ZERO
        else:
            w = ps[K]
        u1 = uniform(b, n, 1)
        y, nt = inverse_cdf(w, u1)
        snear[b] = nt
        final.append((w, u1))
        accepted[b] = n
        out[b, :n] = toks[b, :n]
        out[b, n] = y
        near[b] = path_near
    return ChainResult(accepted, out, mass, near, status, near_rows, snear,
                       final)
