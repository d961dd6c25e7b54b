"""Pins of the EAGLE-2 expand / rerank oracle (EAGLE-2 notes §4.1-§4.2).

* A hand-derived tree in which both tie rules act: equal values at the same
  depth (candidate order), and a child whose draft confidence is exactly 1
  (equal to its parent's value, so the shallower parent must come first,
  which keeps the reranked set connected).
* On random rows: values recomputed with scipy's log_softmax (an independent
  library routine), children = top-k by numpy's stable argsort, layer keep and
  rerank checked by brute force over all candidates, connectivity and
  parent-before-child order.
"""

import math

import numpy as np
from scipy.special import log_softmax

from oracle.eagle2 import expand_rerank
from oracle.tree import tree_mask

NEG = -np.inf


def test_hand_derived_tree_with_ties():
    # V = 4, T = 1, depth 2, 2 children per expanded node, keep 2, total 4.
    # row 0: logits [1, 1, 0, -inf] -> tokens 0 and 1 tie (value v1 each);
    # row 1 (node A = token 0): one-hot on token 0 -> child C keeps value v1
    #   (log 1 = 0), child D has q = 0 -> value -inf;
    # row 2 (node B = token 1): [0, 0, -inf, -inf] -> E, F at v1 - ln 2.
    # Rerank by (value desc, depth asc, id asc): A, B, C, E.
    d = np.array([[[1, 1, 0, NEG],
                   [0, NEG, NEG, NEG],
                   [0, 0, NEG, NEG]]], dtype=np.float64)
    res = expand_rerank(d, temperature=1.0, depth=2, topk=2, width=2,
                        total=4)
    v1 = 1 - math.log(2 * math.e + 1)
    assert list(res.node_tokens[0]) == [0, 1, 0, 0]
    assert list(res.parent[0]) == [-1, -1, 0, 1]
    assert list(res.q_row[0]) == [0, 1, 2, -1, -1]
    assert np.allclose(res.value[0], [v1, v1, v1, v1 - math.log(2)],
                       rtol=0, atol=1e-15)
    want_mask = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 0, 1, 0],
                          [0, 1, 0, 1]], dtype=np.uint8)
    assert np.array_equal(res.mask[0], want_mask)


def _check_random(B, V, T, L, K, W, M, seed):
    rng = np.random.default_rng(seed)
    R = 1 + (L - 1) * W
    d = rng.normal(0, 2.5, (B, R, V)).astype(np.float32).astype(np.float64)
    res = expand_rerank(d, temperature=T, depth=L, topk=K, width=W, total=M)
    for b in range(B):
        lq = log_softmax(d[b] / T, axis=1)
        cands = res.candidates[b]
        # children of every expanded row are its top-K by stable argsort
        rows = {}
        for c in cands:
            par = c["parent"]
            row = 0 if par is None else par["row"]
            rows.setdefault(row, []).append(c)
        for row, kids in rows.items():
            want = list(np.argsort(-d[b, row], kind="stable")[:K])
            assert [c["token"] for c in kids] == want
            for c in kids:
                base = 0.0 if c["parent"] is None else c["parent"]["value"]
                assert abs(c["value"] - (base + lq[row, c["token"]])) < 1e-9
        # layer keep: expanded nodes are the top-W of their layer
        for dep in range(1, L):
            layer = [c for c in cands if c["depth"] == dep]
            ranked = sorted(layer, key=lambda c: (-c["value"], c["id"]))
            kept = [c for c in layer if c["row"] is not None]
            assert sorted(kept, key=lambda c: c["row"]) == ranked[:W]
        # rerank: the selected values are the M best under the tie rule
        key = sorted(cands, key=lambda c: (-c["value"], c["depth"], c["id"]))
        assert [c["token"] for c in key[:M]] == list(res.node_tokens[b])
        # connectivity and order
        for j in range(M):
            pj = res.parent[b, j]
            assert -1 <= pj < j
        m2, _ = tree_mask(res.parent[b:b + 1])
        assert np.array_equal(m2[0], res.mask[b])
        # q_row points at the expansion row of expanded nodes
        for j in range(M):
            r = res.q_row[b, j + 1]
            if r >= 0:
                assert res.node_tokens[b, j] == [c for c in cands
                                                 if c["row"] == r][0]["token"]


def test_random_small_config():
    _check_random(B=3, V=40, T=0.8, L=4, K=3, W=3, M=12, seed=1)


def test_random_eagle2_shape_small_vocab():
    # the shape of the EAGLE-2 workload (depth 6, 10 children, keep 10,
    # total 60) on a small vocabulary
    _check_random(B=2, V=64, T=0.8, L=6, K=10, W=10, M=60, seed=2)
