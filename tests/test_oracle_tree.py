"""Pins of the tree mask and the tree verifier.

* Mask: brute-force ancestor sets; the chain reduces to the lower-triangular
  causal mask (EAGLE-2 notes §4.2).
* Sibling recursion: exact rational enumeration shows the emitted token is
  distributed as p for 1..4 children drawn without replacement (the exactness
  requirement of every page), on the 2-level x 3-children tree of the
  "投机解码与 EAGLE" exercise 4 and the [2, 2, 2] tree of the EAGLE-3 lesson's
  exercise 3.
* verify_tree: Monte-Carlo marginals, and the chain special case equals
  verify_chain decision for decision.
"""

import itertools
from fractions import Fraction as F

import numpy as np
import pytest
from scipy import stats

from oracle.chain import verify_chain
from oracle.sampling import (accept_prob, residual, transform_logits,
                             without_token)
from oracle.tree import tree_mask, verify_tree


def test_mask_brute_force_random_trees():
    rng = np.random.default_rng(0)
    B, N = 6, 23
    parent = np.full((B, N), -1)
    for b in range(B):
        for j in range(N):
            parent[b, j] = int(rng.integers(-1, j)) if j else -1
    mask, bits = tree_mask(parent)
    for b in range(B):
        for i in range(N):
            anc = {i}
            a = parent[b, i]
            while a >= 0:
                anc.add(int(a))
                a = parent[b, a]
            row = {j for j in range(N) if mask[b, i, j]}
            assert row == anc
            assert int(bits[b, i]) == sum(1 << j for j in anc)


def test_mask_chain_is_lower_triangular():
    N = 9
    parent = np.arange(-1, N - 1).reshape(1, N)
    mask, _ = tree_mask(parent)
    assert np.array_equal(mask[0], np.tril(np.ones((N, N), dtype=np.uint8)))


def test_mask_star_is_identity():
    mask, _ = tree_mask(np.full((1, 7), -1))
    assert np.array_equal(mask[0], np.eye(7, dtype=np.uint8))


def _node_law(p, q, m):
    """Exact law of the token emitted at a node with m children drawn from q
    without replacement, built from the oracle's accept_prob / residual /
    without_token helpers."""
    V = len(p)
    out = [F(0)] * V
    if m == 0 or q is None:
        return list(p)
    for x in range(V):
        if q[x] == 0:
            continue
        a = accept_prob(p, q, x)
        out[x] += q[x] * a
        if a == 1:
            continue
        p2, _ = residual(p, q)
        q2 = without_token(q, x)
        sub = _node_law(p2, q2, m - 1) if q2 is not None else list(p2)
        for y in range(V):
            out[y] += q[x] * (1 - a) * sub[y]
    return out


def _rand_dist(rng, V, zero=0.0):
    a = rng.integers(1, 7, V)
    a[rng.random(V) < zero] = 0
    if a.sum() == 0:
        a[0] = 1
    return np.array([F(int(x), int(a.sum())) for x in a], dtype=object)


@pytest.mark.parametrize("m", [1, 2, 3, 4])
def test_sibling_recursion_exact(m):
    rng = np.random.default_rng(m)
    for _ in range(25):
        V = int(rng.integers(2, 5))
        p = _rand_dist(rng, V, zero=0.25)
        q = _rand_dist(rng, V, zero=0.25)
        assert _node_law(p, q, m) == list(p)


def _tree_law(ps, qs, shape, depth=0):
    """Exact law of the first emitted token of a complete tree whose node
    distributions are ps/qs (lists indexed by depth) and branching ``shape``."""
    return _node_law(ps[depth], qs[depth], shape[depth])


@pytest.mark.parametrize("shape", [(3, 3), (2, 2, 2)])
def test_exercise_trees_exact(shape):
    # Every level of the tree runs the same node rule, so the exact law of the
    # token emitted at each node is p for that node's row.
    rng = np.random.default_rng(len(shape))
    V = 4
    for _ in range(10):
        ps = [_rand_dist(rng, V, 0.2) for _ in shape]
        qs = [_rand_dist(rng, V, 0.2) for _ in shape]
        for d in range(len(shape)):
            assert _tree_law(ps, qs, shape, d) == list(ps[d])


def _draw_without_replacement(rng, q, m):
    q = q.copy()
    out = []
    for _ in range(m):
        x = int(rng.choice(q.size, p=q / q.sum()))
        out.append(x)
        q[x] = 0
    return out


def test_tree_monte_carlo_marginals():
    # root with 3 children, each with 2 children ("2 levels" tree)
    V, n = 5, 40_000
    rng = np.random.default_rng(17)
    parent = [-1, -1, -1, 0, 0, 1, 1, 2, 2]
    N = len(parent)
    tl = rng.normal(0, 2, (N + 1, V))
    dl = tl + rng.normal(0, 0.8, (N + 1, V))
    ps = [transform_logits(tl[r], 1.0)[0] for r in range(N + 1)]
    qs = [transform_logits(dl[r], 1.0)[0] for r in range(N + 1)]
    toks = np.zeros((n, N), dtype=np.int64)
    for b in range(n):
        kids = {r: [j for j in range(N) if parent[j] == r - 1]
                for r in range(N + 1)}
        for r, ks in kids.items():
            if ks:
                for j, x in zip(ks, _draw_without_replacement(
                        rng, qs[r], len(ks))):
                    toks[b, j] = x
    res = verify_tree(np.broadcast_to(tl, (n, N + 1, V)),
                      np.broadcast_to(dl, (n, N + 1, V)),
                      np.broadcast_to(np.arange(N + 1), (n, N + 1)), toks,
                      np.broadcast_to(np.array(parent), (n, N)),
                      temperature=1.0, seed=8)
    cnt = np.bincount(res.tokens[:, 0], minlength=V)
    assert stats.chisquare(cnt, ps[0] * n).pvalue > 1e-3
    # second token given the path entered drafted node j
    for j in range(3):
        sel = res.path_nodes[:, 0] == j
        c2 = np.bincount(res.tokens[sel, 1], minlength=V)
        assert stats.chisquare(c2, ps[j + 1] * c2.sum()).pvalue > 1e-3
    for r in range(N + 1):
        assert np.allclose(res.mass[:, r], np.minimum(ps[r], qs[r]).sum())
    # path nodes are consistent with the parent array
    for b in range(200):
        L = res.path_len[b]
        for i in range(L):
            want_parent = res.path_nodes[b, i - 1] if i else -1
            assert parent[res.path_nodes[b, i]] == want_parent


def test_tree_chain_special_case_equals_chain():
    rng = np.random.default_rng(23)
    B, K, V = 40, 5, 11
    tl = rng.normal(0, 2, (B, K + 1, V))
    dl = tl[:, :K] + rng.normal(0, 1.2, (B, K, V))
    toks = rng.integers(0, V, (B, K))
    for kw in (dict(temperature=1.0), dict(temperature=0.6, top_k=5,
                                           top_p=0.8)):
        ch = verify_chain(tl, dl, toks, seed=4, **kw)
        parent = np.broadcast_to(np.arange(-1, K - 1), (B, K))
        qrow = np.broadcast_to(np.r_[np.arange(K), -1], (B, K + 1))
        tr = verify_tree(tl, dl, qrow, toks, parent, seed=4, **kw)
        assert np.array_equal(ch.accepted, tr.path_len)
        assert np.array_equal(ch.tokens, tr.tokens[:, :K + 1])
        assert np.allclose(ch.mass, tr.mass[:, :K])
    ch = verify_chain(tl, None, toks, temperature=0.0)
    tr = verify_tree(tl, None, np.full((B, K + 1), -1), toks,
                     np.broadcast_to(np.arange(-1, K - 1), (B, K)),
                     temperature=0.0)
    assert np.array_equal(ch.accepted, tr.path_len)
    assert np.array_equal(ch.tokens, tr.tokens)


def test_tree_greedy_picks_the_matching_child():
    V = 6
    tl = np.zeros((1, 4, V))
    tl[0, 0, 4] = 3.0   # root argmax 4
    tl[0, 2, 1] = 2.0   # after node 1 (token 4): argmax 1
    parent = np.array([[-1, -1, 1]])
    toks = np.array([[2, 4, 1]])
    res = verify_tree(tl, None, np.full((1, 4), -1), toks, parent,
                      temperature=0.0)
    assert res.path_len[0] == 2
    assert list(res.path_nodes[0, :2]) == [1, 2]
    assert list(res.tokens[0]) == [4, 1, 0, -1]   # row 3 all-zero -> 0
    assert res.mass[0, 0] == 1.0 and res.mass[0, 2] == 1.0


def test_tree_children_without_draft_row_are_flagged():
    rng = np.random.default_rng(1)
    tl = rng.normal(0, 1, (1, 2, 5))
    res = verify_tree(tl, tl, np.array([[-1, -1]]), np.array([[0]]),
                      np.array([[-1]]), temperature=1.0)
    assert res.status & 32 and res.path_len[0] == 0
