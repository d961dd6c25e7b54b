"""Acceptance analytics over verification outcomes (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Three records that the pages ask a deployment to keep about its verifier:

* the distribution of the accepted length per verification round, not only
  its mean ("064 · 投机解码", section 五: two workloads with the same mean
  acceptance can differ in how long runs are);
* the acceptance rate of drafted tokens at each position of the draft tree
  (EAGLE-2 notes §3.1 and Fig. 5: position in the tree, and depth);
* the mean acceptance rate per interval of the draft model's confidence in
  its token (EAGLE-2 notes §3.2 and Fig. 6: confidence below 0.05 is
  accepted about 4% of the time, above 0.95 about 98%).

An acceptance rate is accepted / tested, so each drafted token of a round is
either tested (the verifier took an accept-or-reject decision on it) or not.
The rule that decides (tree verification, EAGLE-2 notes §2.2, with siblings
tried in node order) gives, from the round's outcome alone:

* the accepted tokens are the path's nodes;
* a drafted node is tested iff its parent is the root or on the path, and no
  sibling before it (lower node index) was accepted, i.e. its index is at
  most that of the parent's accepted child (all children of the path's last
  node are tested).

Reading taken: the sequential rule stops trying siblings early in one case,
when the draft distribution has no mass left after removing the rejected
siblings' tokens; the outcome (path) does not show it, and those siblings are
counted as tested.  A chain is the tree whose node k has parent k - 1: token
k is tested iff k <= accepted and accepted iff k < accepted.

The depth of a drafted node is 1 for a child of the root, else its parent's
depth + 1.  Confidence bins: c is clamped to [0, 1] and falls in bin
floor(c * nbins) (the top edge in the last bin), with the product rounded to
float32 as the kernel computes it; a NaN confidence is counted nowhere in the
calibration record.  A round whose outcome is not a root path of its tree
(a count outside [0, n], a node out of range, a node whose parent is not the
previous path node, or a parent array that does not point to earlier nodes)
counts as invalid and adds nothing else.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Stats:
    len_hist: np.ndarray        # [n+1] rounds by accepted length
    node_tested: np.ndarray     # [n]   by node index (chain: position)
    node_accepted: np.ndarray   # [n]
    depth_tested: np.ndarray    # [n]   index = depth - 1
    depth_accepted: np.ndarray  # [n]
    calib_tested: np.ndarray    # [nbins]
    calib_accepted: np.ndarray  # [nbins]
    calib_conf_sum: np.ndarray  # [nbins] float64 sum of clamped confidences
    invalid: int


def empty(n, nbins):
    z = lambda k: np.zeros(k, dtype=np.int64)
    return Stats(z(n + 1), z(n), z(n), z(n), z(n), z(nbins), z(nbins),
                 np.zeros(nbins, dtype=np.float64), 0)


def conf_bin(c, nbins):
    """Bin of confidence c (None for NaN), float32 product as stated."""
    c = np.float32(c)
    if np.isnan(c):
        return None
    c = min(max(c, np.float32(0.0)), np.float32(1.0))
    k = int(np.floor(np.float32(c) * np.float32(nbins)))
    return min(k, nbins - 1), float(c)


def _tree_of(parent_row, n):
    """Parent list of one round (chain when parent_row is None)."""
    if parent_row is None:
        return [k - 1 for k in range(n)]
    return [int(x) for x in parent_row]


def round_outcome(par, length, path):
    """(tested, accepted) node sets of one round, or None if invalid."""
    n = len(par)
    if any(not -1 <= par[j] < j for j in range(n)):
        return None
    if not 0 <= length <= n:
        return None
    prev = -1
    for i in range(length):
        v = int(path[i])
        if not 0 <= v < n or par[v] != prev:
            return None
        prev = v
    on_path = [int(path[i]) for i in range(length)]
    # the accepted child of the root and of every path node (None: none)
    acc_child = {-1: on_path[0] if length else None}
    for i, v in enumerate(on_path):
        acc_child[v] = on_path[i + 1] if i + 1 < length else None
    tested = set()
    for j in range(n):
        if par[j] in acc_child:
            a = acc_child[par[j]]
            if a is None or j <= a:
                tested.add(j)
    return tested, set(on_path)


def depths(par):
    d = []
    for j in range(len(par)):
        d.append(1 if par[j] < 0 else d[par[j]] + 1)
    return d


def accept_stats(count, parent, path_nodes, confidence, n, nbins=20,
                 into=None):
    """Add one batch of rounds to the records.

    count [B]: accepted drafts (chain) or path length (tree).  parent [B, n]
    and path_nodes [B, n] for a tree, both None for a chain.  confidence
    [B, n] or None.  Returns the Stats (``into`` updated in place if given).
    """
    st = into if into is not None else empty(n, nbins)
    B = len(count)
    for b in range(B):
        par = _tree_of(None if parent is None else parent[b], n)
        L = int(count[b])
        path = list(range(L)) if path_nodes is None else path_nodes[b]
        if path_nodes is None and not 0 <= L <= n:
            st.invalid += 1
            continue
        res = round_outcome(par, L, path)
        if res is None:
            st.invalid += 1
            continue
        tested, accepted = res
        st.len_hist[L] += 1
        dep = depths(par)
        for j in sorted(tested):
            ok = j in accepted
            st.node_tested[j] += 1
            st.node_accepted[j] += ok
            st.depth_tested[dep[j] - 1] += 1
            st.depth_accepted[dep[j] - 1] += ok
            if confidence is not None:
                cb = conf_bin(confidence[b][j], nbins)
                if cb is None:
                    continue
                k, c = cb
                st.calib_tested[k] += 1
                st.calib_accepted[k] += ok
                st.calib_conf_sum[k] += c
    return st
