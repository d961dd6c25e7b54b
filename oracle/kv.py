"""KV-cache commit after verification (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The verification pass runs the target model over every drafted position at
once, so it appends one KV entry per drafted position after the committed
prefix.  Afterwards only the accepted drafts may stay in the cache:

* "Việc giải mã giả định và EAGLE-3", section "KV cache rollback": the
  verifier's cache grows by the number of drafts; after a rejection it must
  hold only the accepted prefix.  Of the two usual implementations (a scratch
  buffer committed on acceptance, or one physical cache plus a logical length
  cut back on rejection) the chain case here is the second: nothing moves,
  the logical length becomes prefix + accepted.  Its step 4 ("kế toán KV")
  keeps exactly that logical length.
* "Descodación especulativa Draft, Verificar, Replicar", section "El baile
  de caché KV" and its exercise 4: after a rejection the next iteration must
  read the prefix plus the accepted drafts, and nothing of the rejected ones.

A tree (EAGLE-2 notes §4.2) writes drafted node j's entry at position
prefix + j in node order; the accepted path is a subsequence of the nodes, so
committing it means moving path node i's entry to position prefix + i.  Read
plainly: for i = 0, 1, ..., in path order, copy position prefix + node_i to
position prefix + i.  The path's nodes increase (parents precede children),
so node_i >= i and the in-place copy never overwrites an entry it still has
to read; ``kv_commit_gather`` states the same result without aliasing and the
tests compare the two.

The token drawn after the path has no entry yet: the next forward pass
writes it.  New logical length = prefix + path length.
"""

import numpy as np


def path_valid(nodes, length, n):
    """A path the commit accepts: 0 <= length <= n, nodes strictly
    increasing inside [0, n)."""
    if length < 0 or length > n:
        return False
    prev = -1
    for i in range(length):
        v = int(nodes[i])
        if v <= prev or v >= n:
            return False
        prev = v
    return True


def kv_commit(cache, prefix_len, path_len, path_nodes=None, n=None):
    """Commit the accepted drafts of every sequence.

    cache: array [B, S, ...] (position axis 1, any trailing shape); a copy is
    changed and returned.  prefix_len, path_len: [B] ints.  path_nodes:
    [B, n] ints (tree) or None (chain: the accepted drafts are already the
    first positions after the prefix).  Returns (cache', new_len) with
    new_len[b] = prefix + path_len, or -1 (sequence left unchanged) for an
    invalid path."""
    out = np.array(cache, copy=True)
    B = out.shape[0]
    new_len = np.empty(B, dtype=np.int64)
    for b in range(B):
        pre, length = int(prefix_len[b]), int(path_len[b])
        if path_nodes is None:
            ok = 0 <= length <= (n if n is not None else length)
            new_len[b] = pre + length if ok else -1
            continue
        nodes = path_nodes[b]
        if not path_valid(nodes, length, path_nodes.shape[1]):
            new_len[b] = -1
            continue
        for i in range(length):  # in path order, in place
            out[b, pre + i] = out[b, pre + int(nodes[i])]
        new_len[b] = pre + length
    return out, new_len


def kv_commit_gather(cache, prefix_len, path_len, path_nodes):
    """The tree commit stated without aliasing: positions prefix + i of the
    result take the ORIGINAL entry of position prefix + node_i; every other
    position keeps its original entry.  Valid paths only."""
    out = np.array(cache, copy=True)
    src = np.array(cache, copy=True)
    for b in range(out.shape[0]):
        pre, length = int(prefix_len[b]), int(path_len[b])
        for i in range(length):
            out[b, pre + i] = src[b, pre + int(path_nodes[b][i])]
    return out
