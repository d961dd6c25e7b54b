"""Pins of the acceptance-analytics oracle (no GPU).

The records follow "064 · 投机解码" section 五 (accepted-length distribution)
and the EAGLE-2 notes §3.1 / §3.2 (acceptance rate by tree position and by
draft-confidence interval).  They are pinned by a hand-worked example, by an
exhaustive comparison with a step-by-step simulation of the verifier's
decisions, by the closed forms of an i.i.d. chain, by a calibrated drafter,
and by the exact acceptance probabilities of the first and second sibling
under the tree verification rule.
"""

import math
import os

import numpy as np
import pytest

from oracle import stats
from oracle.analysis import expected_tokens
from oracle.sampling import acceptance_mass, residual, transform, without_token
from oracle.tree import verify_tree

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "accept_stats_example.txt")


def _golden():
    rec = {}
    for ln in open(GOLDEN, encoding="utf-8"):
        if not ln.strip() or ln.startswith("#"):
            continue
        parts = ln.split()
        rec[(parts[0], parts[1])] = parts[2:]
    return rec


def test_hand_worked_tree_example():
    g = _golden()
    parent = [int(x) for x in g[("tree", "parent")]]
    n = len(parent)
    # several "path" lines share a key: read them in file order
    paths = []
    for ln in open(GOLDEN, encoding="utf-8"):
        p = ln.split()
        if p[:2] == ["tree", "path"]:
            paths.append([int(x) for x in p[3:]])
    conf = [float(x) for x in g[("tree", "conf")]]
    nbins = int(g[("tree", "nbins")][0])
    B = len(paths)
    count = [len(p) for p in paths]
    nodes = np.full((B, n), -1)
    for b, p in enumerate(paths):
        nodes[b, :len(p)] = p
    st = stats.accept_stats(count, np.tile(parent, (B, 1)), nodes,
                            np.tile(np.float32(conf), (B, 1)), n, nbins)
    for name in ("len_hist", "node_tested", "node_accepted", "depth_tested",
                 "depth_accepted", "calib_tested", "calib_accepted"):
        want = [int(x) for x in g[("tree", name)]]
        assert list(getattr(st, name)) == want, name
    assert st.invalid == int(g[("tree", "invalid")][0])
    f = lambda x: float(np.float32(x))
    want_sum = [0.0, 2 * f(0.3) + 0.25, 2 * f(0.6), 4 * f(0.9) + 1.0]
    assert np.allclose(st.calib_conf_sum, want_sum, rtol=0, atol=1e-15)


def test_hand_worked_chain_example():
    g = _golden()
    n = int(g[("chain", "n")][0])
    count = [int(x) for x in g[("chain", "count")]]
    st = stats.accept_stats(count, None, None, None, n)
    for name in ("len_hist", "node_tested", "node_accepted"):
        assert list(getattr(st, name)) == [int(x) for x in g[("chain", name)]]
    # chain: depth k + 1 is position k
    assert np.array_equal(st.depth_tested, st.node_tested)
    assert st.invalid == int(g[("chain", "invalid")][0])


def _random_tree(rng, n):
    return [-1 if j == 0 or rng.random() < 0.3 else int(rng.integers(0, j))
            for j in range(n)]


def _simulate(par, decide):
    """The verifier's decisions, one by one: from the root, try the children
    in node order; an accepted child becomes the current node; stop when all
    children of the current node are rejected or it has none.  Returns the
    path and the (node, accepted) decisions in the order they were taken."""
    n = len(par)
    kids = {v: [j for j in range(n) if par[j] == v] for v in range(-1, n)}
    cur, path, log = -1, [], []
    while True:
        nxt = None
        for j in kids[cur]:
            ok = decide(j)
            log.append((j, ok))
            if ok:
                nxt = j
                break
        if nxt is None:
            return path, log
        path.append(nxt)
        cur = nxt


def test_tested_set_equals_step_by_step_decisions_exhaustively():
    # every accept/reject assignment of small trees, including the [2,2,2]
    # tree of the Vietnamese lesson and a chain
    rng = np.random.default_rng(3)
    trees = [[-1, -1, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5],  # [2,2,2]: 14 nodes
             [-1, 0, 1, 2, 3], [-1, -1, -1, 0, 0, 1, 4]]
    trees += [_random_tree(rng, int(rng.integers(1, 11))) for _ in range(12)]
    for par in trees:
        n = len(par)
        dep = stats.depths(par)
        for mask in range(1 << n):
            decide = lambda j: bool(mask >> j & 1)
            path, log = _simulate(par, decide)
            res = stats.round_outcome(par, len(path), path)
            assert res is not None
            tested, acc = res
            assert tested == {j for j, _ in log}
            assert acc == {j for j, ok in log if ok}
            st = stats.accept_stats([len(path)], [par],
                                    [path + [-1] * (n - len(path))], None, n)
            assert st.len_hist[len(path)] == 1 and st.len_hist.sum() == 1
            for j, ok in log:
                assert st.node_tested[j] == 1 and st.node_accepted[j] == ok
            assert st.depth_tested.sum() == len(log)
            assert st.depth_accepted.sum() == len(path)
            assert all(dep[v] == i + 1 for i, v in enumerate(path))


def test_invalid_rounds_add_nothing_else():
    par = [-1, -1, 0, 1]
    cases = [(3, [0, 2, 3]),   # 3 is not a child of 2
             (1, [2]),         # 2 is not a child of the root
             (5, [0, 2]),      # count above n
             (-1, []),         # negative count
             (1, [7])]         # node out of range
    for L, path in cases:
        nodes = np.full((1, 4), -1)
        nodes[0, :len(path)] = path[:4]
        st = stats.accept_stats([L], [par], nodes, [[0.5] * 4], 4, 4)
        assert st.invalid == 1
        assert st.len_hist.sum() == 0 and st.node_tested.sum() == 0
        assert st.calib_tested.sum() == 0
    # a parent array that points forward is invalid too
    st = stats.accept_stats([0], [[1, -1]], [[-1, -1]], None, 2)
    assert st.invalid == 1


def test_iid_chain_matches_closed_forms():
    # i.i.d. acceptance at rate alpha, K = 4: accepted length is a truncated
    # geometric, E[tokens] = (1 - a^(K+1)) / (1 - a) = 3.3616 at a = 0.8
    # ("投机解码与 EAGLE", 期望加速比), and every position's rate is alpha
    rng = np.random.default_rng(5)
    a, K, B = 0.8, 4, 200_000
    acc = rng.random((B, K)) < a
    count = np.where(acc.all(axis=1), K, np.argmin(acc, axis=1))
    st = stats.accept_stats(count[:20000], None, None, None, K)
    # the remaining rounds added into the same record, batch by batch
    for lo in range(20000, B, 20000):
        stats.accept_stats(count[lo:lo + 20000], None, None, None, K, into=st)
    h = st.len_hist / B
    want = [a ** L * (1 - a) for L in range(K)] + [a ** K]
    for L in range(K + 1):
        sd = math.sqrt(want[L] * (1 - want[L]) / B)
        assert abs(h[L] - want[L]) < 5 * sd
    mean_tokens = float((np.arange(K + 1) + 1) @ st.len_hist) / B
    assert abs(mean_tokens - expected_tokens(a, K)) < 0.01
    assert abs(expected_tokens(a, K) - 3.3616) < 1e-12
    for k in range(K):
        assert st.node_tested[k] == int((count >= k).sum())
        rate = st.node_accepted[k] / st.node_tested[k]
        assert abs(rate - a) < 5 * math.sqrt(a * (1 - a) / st.node_tested[k])


def test_calibrated_drafter_sits_on_the_diagonal():
    # a drafter whose token is accepted with probability equal to its
    # confidence: every interval's rate is its mean confidence (Fig. 6's
    # dashed diagonal); one squaring the confidence falls below it
    rng = np.random.default_rng(6)
    K, B, nb = 3, 40_000, 10
    for power in (1, 2):
        conf = rng.random((B, K)).astype(np.float32)
        acc = rng.random((B, K)) < conf.astype(np.float64) ** power
        count = np.where(acc.all(axis=1), K, np.argmin(acc, axis=1))
        st = stats.accept_stats(count, None, None, conf, K, nb)
        for k in range(nb):
            t = st.calib_tested[k]
            assert t > 1000
            mean_c = st.calib_conf_sum[k] / t
            assert k / nb <= mean_c < (k + 1) / nb
            rate = st.calib_accepted[k] / t
            lo, hi = (k / nb) ** power, ((k + 1) / nb) ** power
            sd = math.sqrt(0.25 / t)
            assert lo - 5 * sd < rate < hi + 5 * sd
            if power == 1:
                assert abs(rate - mean_c) < 5 * sd


def test_confidence_bins_at_the_edges():
    nb = 20
    assert stats.conf_bin(0.05, nb)[0] == 1     # 0.05f * 20 rounds to 1.0
    assert stats.conf_bin(1.0, nb)[0] == nb - 1
    assert stats.conf_bin(0.0, nb)[0] == 0
    assert stats.conf_bin(-3.0, nb) == (0, 0.0)
    assert stats.conf_bin(7.0, nb) == (nb - 1, 1.0)
    assert stats.conf_bin(float("nan"), nb) is None
    below = float(np.nextafter(np.float32(0.5), np.float32(0)))
    assert stats.conf_bin(below, 2)[0] == 0 and stats.conf_bin(0.5, 2)[0] == 1


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.slow
def test_sibling_rates_match_the_tree_rule_exactly():
    # Tree: two children of the root (node 0, node 1), sibling tokens drawn
    # without replacement from q (as the static-tree inputs are).  Under the
    # tree verification rule the first child is accepted with probability
    # alpha = sum min(p, q); given its rejection the second child's rate is
    # sum over x1 of P(x1 | rejected) * sum min(p', q'_{-x1}).  The records
    # computed from verify_tree's outcomes must reproduce both.
    rng = np.random.default_rng(8)
    V, B = 6, 6000
    zt = rng.normal(0, 1.0, V)
    q = _softmax(zt + rng.normal(0, 0.9, V))
    p, _ = transform(zt, "logits", 1.0, 0, 1.0)
    alpha = acceptance_mass(p, q)
    a1 = np.minimum(1.0, p / q)
    rej = q * (1 - a1)
    second = 0.0
    pr, _ = residual(p, q)
    for x1 in range(V):
        qm = without_token(q, x1)
        second += rej[x1] / rej.sum() * acceptance_mass(pr, qm)
    parent = np.tile([-1, -1], (B, 1))
    toks = np.empty((B, 2), dtype=np.int32)
    for b in range(B):
        toks[b] = rng.choice(V, size=2, replace=False, p=q)
    target = np.tile(zt, (B, 3, 1))
    draft = np.tile(q, (B, 1, 1))
    q_row = np.tile([0, -1, -1], (B, 1))
    res = verify_tree(target, draft, q_row, toks, parent, temperature=1.0,
                      draft_kind="probs", seed=9)
    st = stats.accept_stats(res.path_len, parent, res.path_nodes, None, 2)
    assert st.node_tested[0] == B
    r0 = st.node_accepted[0] / B
    assert abs(r0 - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / B)
    t1 = st.node_tested[1]
    assert t1 == B - st.node_accepted[0]
    r1 = st.node_accepted[1] / t1
    assert abs(r1 - second) < 5 * math.sqrt(second * (1 - second) / t1)
    assert st.len_hist[1] == st.node_accepted.sum()
