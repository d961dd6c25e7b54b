"""Tree attention of the verification pass (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

EAGLE-2 notes §4.2 (constructing the verification input and its attention
mask): the selected draft tokens are flattened into one sequence and run
through the target model in one pass; in plain decoding every token sees all
earlier tokens (a lower-triangular mask), but tokens of different branches
must not see each other, so each drafted token sees only its ancestors.  The
Spanish lesson's Medusa section verifies all candidate continuations in one
pass with the same tree attention.

So for sequence b with committed prefix length P (its keys and values already
in the cache at positions 0 .. P-1) and drafted node i (its key and value at
position P + i, its query q_i), in every query head h:

    visible(i) = {0 .. P-1} + {P + j : j = i or j an ancestor of i}
    o_i = sum_{s in visible(i)} softmax_s(scale * q_i . k_s) v_s

with the softmax over visible(i) only.  Grouped-query attention: query head h
reads key/value head h // (Hq / Hkv).  Computed here in float64 from the
given (bf16-valued) inputs.
"""

from __future__ import annotations

import numpy as np

from .tree import ancestors


def visible_keys(parent_row, i, P):
    """Key positions drafted node i attends to (prefix first, then its
    ancestors and itself in position order)."""
    tree = sorted(ancestors(parent_row, i) | {i})
    return list(range(P)) + [P + j for j in tree]


def tree_attention(q, k, v, prefix_len, parent, scale):
    """q [B, N, Hq, D]; k, v [B, Hkv, S, D]; prefix_len [B]; parent [B, N].
    Returns o [B, N, Hq, D] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, N, Hq, D), dtype=np.float64)
    for b in range(B):
        P = int(prefix_len[b])
        for i in range(N):
            keys = visible_keys(parent[b], i, P)
            for h in range(Hq):
                kv = h // G
                s = scale * (k[b, kv, keys] @ q[b, i, h])
                w = np.exp(s - s.max())
                w /= w.sum()
                out[b, i, h] = w @ v[b, kv, keys]
    return out
