"""Tree attention mask and tree verification (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Layout.  A draft tree has N drafted nodes j = 0 .. N-1 with tokens t_j and a
parent array: parent[j] = -1 for a child of the root (the last committed
position) and parent[j] in [0, j) otherwise (parents precede children, as the
flattened order of the EAGLE-2 notes §4.2 gives).  Target row r = 0 is the
root; row r = j + 1 is the position after drafted node j.  ``q_row[r]`` names
the draft row holding q at tree row r, or -1.

Mask (EAGLE-2 notes §4.2, the paragraph on the verification input and
its attention mask): drafted token i
sees drafted token j iff j is an ancestor of i or i itself (the chain case is
the lower-triangular causal mask); the committed prefix is visible to all and
is not part of the N x N mask.

Verification.  A tree lets a rejected branch give way to its siblings
(EAGLE-2 notes §2.2, the verification stage of tree drafts).  The pages do not
spell the multi-sibling rule out; we take the lossless reading that the
exactness requirement of every page forces: recursive rejection sampling over
the children of a node, tried in node-index order, with siblings drawn
without replacement from q.  At tree row r with children c_1 < ... < c_m:

    p' = p_r, q' = q_r
    for child c_j with token x:
        accept iff u(b, c_j, 0) < p'(x) / q'(x)          (q'(x) = 0 accepts)
        on rejection: p' <- norm(max(0, p' - q'))        (zero mass: keep p')
                      q' <- q' with x removed, renormalised (none left: stop)
    no child accepted: sample the emitted token from p' with u(b, r, 1)
    (a leaf has no children, so this is the bonus draw from p_r).

The walk starts at the root and follows accepted children; the path is the
accepted drafted nodes and the emitted tokens are their tokens followed by the
token sampled at the last node.  With one child per node this is exactly the
chain rule.  Temperature 0: a child is accepted iff its token equals the
argmax of the target logits at its parent's row (first such child in index
order); otherwise the argmax is emitted.

alpha_r = sum_x min(p_r, q_r) for every row with a draft row (NaN otherwise).
At temperature 0 both distributions are point masses, so alpha_r is 1 when a
child of row r matches the argmax and 0 when none does (NaN for a row without
children), which is the chain's 1[x_k == argmax] on a path.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox
from .chain import (ST_BAD_TREE, ST_DRAFT_EXHAUSTED, ST_QZERO_ACCEPT,
                    ST_RESIDUAL_ZERO, ST_TOKEN_RANGE)
from .sampling import (accept, acceptance_mass, argmax_first, inverse_cdf,
                       residual, transform, without_token)


def ancestors(parent, j):
    """Set of drafted-node ancestors of node j (excluding j).  The walk ends
    at the root (-1) or at the first link that does not point to an earlier
    node (an invalid parent array)."""
    out = set()
    cur = j
    a = int(parent[j])
    while 0 <= a < cur:
        out.add(a)
        cur = a
        a = int(parent[a])
    return out


def tree_mask(parent):
    """parent [B, N] -> (mask [B, N, N] uint8, bits [B, N] uint64 or None)."""
    parent = np.asarray(parent)
    B, N = parent.shape
    mask = np.zeros((B, N, N), dtype=np.uint8)
    for b in range(B):
        for i in range(N):
            for j in ancestors(parent[b], i) | {i}:
                mask[b, i, j] = 1
    bits = None
    if N <= 64:
        bits = np.zeros((B, N), dtype=np.uint64)
        for b in range(B):
            for i in range(N):
                v = 0
                for j in range(N):
                    if mask[b, i, j]:
                        v |= 1 << j
                bits[b, i] = np.uint64(v)
    return mask, bits


def valid_parent(parent_row):
    return all(-1 <= int(parent_row[j]) < j for j in range(len(parent_row)))


@dataclass
class TreeResult:
    path_len: np.ndarray      # [B] int32: accepted drafted nodes
    path_nodes: np.ndarray    # [B, N] int32, -1 padded
    tokens: np.ndarray        # [B, N+1] int32, -1 padded
    mass: np.ndarray          # [B, N+1] float64 (NaN where no draft row)
    near_tie: np.ndarray      # [B] bool: accept test / top-p cut near tie
    status: int = 0
    outcome: list = field(default_factory=list)  # per b: {row: child or None}
    sample_near: np.ndarray = None  # [B] bool: final draw near a CDF boundary
    final: list = field(default_factory=list)      # per b: (weights, u)


def verify_tree(target, draft, q_row, node_tokens, parent, *,
                temperature: float, top_k: int = 0, top_p: float = 1.0,
                draft_kind="logits", seed: int = 0, offset: int = 0,
                uniform=None, batch_ids=None) -> TreeResult:
    """target [B, N+1, V], draft [B, R, V] (None at temperature 0),
    q_row [B, N+1], node_tokens [B, N], parent [B, N]."""
    target = np.asarray(target)
    B, N1, V = target.shape
    N = N1 - 1
    q_row = np.asarray(q_row).reshape(B, N + 1)
    toks = np.asarray(node_tokens).reshape(B, N)
    parent = np.asarray(parent).reshape(B, N)
    if uniform is None:
        # batch_ids: the sequence index each row had in the full batch (the
        # Philox counter uses it), when the oracle checks a subset
        ids = list(range(B)) if batch_ids is None else [int(x) for x in
                                                         batch_ids]

        def uniform(b, i, slot):
            return philox.uniform(seed, ids[b], i, slot, offset)

    path_len = np.zeros(B, dtype=np.int32)
    path_nodes = np.full((B, N), -1, dtype=np.int32)
    out = np.full((B, N + 1), -1, dtype=np.int32)
    mass = np.full((B, N + 1), np.nan, dtype=np.float64)
    near = np.zeros(B, dtype=bool)
    snear = np.zeros(B, dtype=bool)
    final = []
    status = 0
    outcomes = []

    for b in range(B):
        if not valid_parent(parent[b]):
            status |= ST_BAD_TREE
        children = {r: [] for r in range(N + 1)}
        for j in range(N):
            pj = int(parent[b, j])
            if -1 <= pj < j:
                children[pj + 1].append(j)
        # per-row outcome: accepted child or the sampled token (+ near flag)
        acc = {}
        tok = {}
        nrow = {}
        draw = {}   # row -> (weights, u, near) of its sampled token
        for r in range(N + 1):
            kids = children[r]
            if temperature == 0:
                g = argmax_first(target[b, r])
                acc[r] = next((j for j in kids if toks[b, j] == g), None)
                tok[r] = g
                nrow[r] = False
                draw[r] = (None, None, False)
                if kids:  # greedy point masses: overlap is 1 iff a child hits
                    mass[b, r] = 1.0 if acc[r] is not None else 0.0
                continue
            p, nt = transform(target[b, r], "logits", temperature, top_k,
                              top_p)
            row_near = nt
            q = None
            if q_row[b, r] >= 0:
                q, nt = transform(np.asarray(draft)[b, q_row[b, r]],
                                  draft_kind, temperature, top_k, top_p)
                row_near |= nt
                mass[b, r] = acceptance_mass(p, q)
            if kids and q is None:
                status |= ST_BAD_TREE
                kids = []
            pc, qc = p, q
            acc[r] = None
            for j in kids:
                x = int(toks[b, j])
                if not 0 <= x < V:
                    status |= ST_TOKEN_RANGE
                    ok, nt, qz = False, False, False
                else:
                    ok, nt, qz = accept(pc, qc, x, uniform(b, j, 0))
                row_near |= nt
                if qz:
                    status |= ST_QZERO_ACCEPT
                if ok:
                    acc[r] = j
                    break
                pc, fb = residual(pc, qc)
                if fb:
                    status |= ST_RESIDUAL_ZERO
                if 0 <= x < V:
                    qc = without_token(qc, x)
                if qc is None:
                    status |= ST_DRAFT_EXHAUSTED
                    break
            if acc[r] is None:
                u1 = uniform(b, r, 1)
                y, nt = inverse_cdf(pc, u1)
                tok[r] = y
                draw[r] = (pc, u1, nt)
            nrow[r] = row_near
        # walk from the root
        r = 0
        path = []
        path_near = nrow[0]
        while acc[r] is not None:
            j = acc[r]
            path.append(j)
            r = j + 1
            path_near |= nrow[r]
        snear[b] = draw[r][2]
        final.append(draw[r][:2])
        path_len[b] = len(path)
        path_nodes[b, :len(path)] = path
        out[b, :len(path)] = [toks[b, j] for j in path]
        out[b, len(path)] = tok[r]
        near[b] = path_near
        outcomes.append({"acc": acc, "tok": tok, "near": nrow})
    return TreeResult(path_len, path_nodes, out, mass, near, status, outcomes,
                      snear, final)
