"""Target LM head of the verification pass, then tree verification (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Step 2 of the draft/verify loop ("投机解码与 EAGLE", the four steps of one
round) runs the target model once over all drafted positions and reads its
next-token distribution at each of them; "064 · 投机解码" (section 二, why the
verification is parallel) says the same of the target's conditional
distributions.  The last layer of that forward pass maps each position's
final hidden state h (the feature EAGLE's drafter reuses, "EAGLE-2" notes
§2.2) to the target logits over the vocabulary: z[v] = sum_h h[h] W[v, h],
with W [V, H] the output embedding (LM head) matrix.  The pages do not write
this layer out; this is the plain reading.

Precision (a reading; the pages are silent): hidden states and W are bf16,
the product is accumulated in float32 and the logits the verifier reads are
rounded to bf16, as a bf16 forward pass produces them (the static-tree
workload's target logits are bf16).  The oracle computes z exactly (float64
products of bf16 values are exact; the sum of H of them is within float64
rounding) and rounds it to bf16 from the format's definition.

Because the device accumulates in float32, its float32 logit lies within
``delta`` of the exact one, and its bf16 logit is the rounding of that value:
any bf16 value from ``lo`` = RN(z - delta) to ``hi`` = RN(z + delta).
``delta`` bounds the float32 accumulation error of H products summed in
groups of 16 with round-to-nearest:

    delta[v] = (H / 16 + 16) * 2^-24 * sum_h |h[h] W[v, h]|.

Away from zero that range is the exact value's two bf16 neighbours at most;
near zero (a sum that cancels) a bf16 unit is far below delta and the range
spans many bf16 values.  Logits with lo != hi are "ambiguous".  The
verification is run on the nearest rounding and on the two ends of the range
(every ambiguous logit at lo, then at hi); a sequence whose decisions (path
and emitted tokens before the final draw) differ between the runs is a
rounding near tie and is excluded from exact comparison, like an accept test
within 1e-5 of its threshold.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .tree import TreeResult, verify_tree


def bf16_neighbours(x):
    """(lo, hi): the bf16 values below and above x (equal when x is a bf16
    value).  bf16 keeps 8 significant bits; for x = m 2^e with
    0.5 <= |m| < 1, the neighbours are floor / ceil of m 2^8 times 2^(e-8).
    Normal-range finite values only (the logits here are far from the
    subnormal and overflow ranges)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    t = m * 256.0
    lo = np.ldexp(np.floor(t), e - 8)
    hi = np.ldexp(np.ceil(t), e - 8)
    return lo, hi


def bf16_round(x):
    """Round to the nearest bf16 value, ties to the one with an even last
    significand bit (IEEE round-to-nearest-even at 8 significant bits)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    # numpy's round is round-half-to-even on the integer m * 2^8
    return np.ldexp(np.round(m * 256.0), e - 8)


@dataclass
class LMHead:
    exact: np.ndarray      # [..., V] float64: sum_h h W (exact up to f64)
    rn: np.ndarray         # [..., V] float64: exact rounded to bf16
    lo: np.ndarray         # [..., V]: RN(exact - delta), the lowest bf16 result
    hi: np.ndarray         # [..., V]: RN(exact + delta), the highest
    ambiguous: np.ndarray  # [..., V] bool: lo != hi
    delta: np.ndarray      # [..., V] the accumulation-error bound used


def lm_head_logits(hidden, w):
    """hidden [..., H], w [V, H] (bf16 values as float64).  Returns the
    LMHead record of the target logits."""
    h = np.asarray(hidden, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    H = h.shape[-1]
    exact = h @ w.T
    delta = (H / 16.0 + 16.0) * 2.0 ** -24 * (np.abs(h) @ np.abs(w).T)
    rn = bf16_round(exact)
    lo = bf16_round(exact - delta)
    hi = bf16_round(exact + delta)
    return LMHead(exact, rn, lo, hi, lo != hi, delta)


@dataclass
class LMHeadTreeResult:
    ref: TreeResult            # verification on the rounded logits
    rounding_tie: np.ndarray   # [B] bool: the other rounding decides otherwise
    logits: LMHead
    mass_slack: np.ndarray = None  # [B, N+1]: bound on the acceptance-mass
                                   # change any rounding in range can cause


def mass_slack(lg, temperature):
    """Per row, a bound on how far alpha = sum min(p, q) can move when the
    logits take any values in [lo, hi] instead of rn (full-vocabulary
    transform at temperature T > 0).  A logit moved by at most d = hi - lo
    scales its unnormalised weight by at most e^(d / T); so p changes by at
    most p (e^(d/T) - 1) at the moved tokens plus the normaliser's relative
    change, which is bounded by the same sum: |d alpha| <= 2 sum_amb p_v
    (e^(d_v / T) - 1)."""
    z = lg.rn / temperature
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    d = np.where(lg.ambiguous, lg.hi - lg.lo, 0.0) / temperature
    return 2.0 * (p * np.expm1(d)).sum(axis=-1)


def verify_tree_lmhead(hidden, w, draft, q_row, node_tokens, parent, **kw):
    """Target logits from the LM head (hidden [B, N+1, H], w [V, H]), then
    tree verification with the keyword arguments of verify_tree.  The
    result's ``ref.near_tie`` includes the rounding near ties."""
    lg = lm_head_logits(hidden, w)
    ref = verify_tree(lg.rn, draft, q_row, node_tokens, parent, **kw)
    B = ref.path_len.shape[0]
    tie = np.zeros(B, dtype=bool)
    if lg.ambiguous.any():
        for end in (lg.lo, lg.hi):
            other = verify_tree(end, draft, q_row, node_tokens, parent, **kw)
            for b in range(B):
                n = int(ref.path_len[b])
                same = (n == int(other.path_len[b]) and
                        np.array_equal(ref.path_nodes[b],
                                       other.path_nodes[b]) and
                        np.array_equal(ref.tokens[b][:n],
                                       other.tokens[b][:n]))
                tie[b] |= not same
    ref.near_tie = ref.near_tie | tie
    T = kw.get("temperature", 0.0)
    slack = mass_slack(lg, T) if T > 0 else None
    return LMHeadTreeResult(ref, tie, lg, slack)
