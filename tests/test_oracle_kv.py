"""Pins of the KV-cache commit oracle (no GPU)."""

import os

import numpy as np
import pytest

from oracle.kv import kv_commit, kv_commit_gather, path_valid
from oracle.tree import verify_tree

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_rollback.txt")


def _rollback_case():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    return [int(x) for x in rows[0]]


def test_rollback_exercise_of_the_spanish_page():
    prefix, drafts, reject_at, accepted, new_len = _rollback_case()
    assert accepted == reject_at - 1  # drafts before the first rejection
    S = prefix + drafts
    # entry payload = the position's token id: prefix tokens 100.., drafts 200..
    cache = np.concatenate([100 + np.arange(prefix), 200 + np.arange(drafts)])
    cache = cache.reshape(1, S, 1)
    out, nl = kv_commit(cache, [prefix], [accepted], None, n=drafts)
    assert nl[0] == new_len
    read = out[0, :nl[0], 0]
    assert list(read) == list(100 + np.arange(prefix)) + [200, 201]


def test_chain_logical_length_closed_form():
    rng = np.random.default_rng(0)
    B, K = 7, 5
    cache = rng.integers(0, 1 << 30, size=(B, 40, 3))
    pre = rng.integers(0, 30, size=B)
    acc = rng.integers(0, K + 1, size=B)
    out, nl = kv_commit(cache, pre, acc, None, n=K)
    assert np.array_equal(nl, pre + acc)      # kv_length += k
    assert np.array_equal(out, cache)          # a chain moves nothing


def _random_path(rng, n, length):
    return np.sort(rng.choice(n, size=length, replace=False))


def test_in_place_path_order_equals_alias_free_gather():
    rng = np.random.default_rng(1)
    for trial in range(200):
        B, n = 4, int(rng.integers(1, 12))
        S = 10 + n
        cache = rng.integers(0, 1 << 30, size=(B, S, 2))
        pre = rng.integers(0, 10, size=B)
        lens = rng.integers(0, n + 1, size=B)
        nodes = np.full((B, n), -1)
        for b in range(B):
            nodes[b, :lens[b]] = _random_path(rng, n, lens[b])
        out, nl = kv_commit(cache, pre, lens, nodes)
        ref = kv_commit_gather(cache, pre, lens, nodes)
        assert np.array_equal(out, ref)
        assert np.array_equal(nl, pre + lens)
        # positions outside [pre, pre + len) are untouched
        for b in range(B):
            keep = np.ones(S, bool)
            keep[pre[b]:pre[b] + lens[b]] = False
            assert np.array_equal(out[b, keep], cache[b, keep])


def test_identity_path_moves_nothing_and_invalid_paths_are_refused():
    cache = np.arange(2 * 12).reshape(2, 12, 1)
    nodes = np.array([[0, 1, 2, -1], [2, 1, -1, -1]])
    out, nl = kv_commit(cache, [3, 3], [3, 2], nodes)
    assert np.array_equal(out, cache)          # 0,1,2 in place; 2,1 refused
    assert list(nl) == [6, -1]
    assert not path_valid([0, 4], 2, 4) and not path_valid([1, 1], 2, 4)
    assert not path_valid([0], 5, 4) and path_valid([], 0, 0)


def test_tree_commit_keeps_the_tokens_verification_emits():
    # payload of node j = its token: after the commit the first path-length
    # entries after the prefix are the accepted tokens verify_tree emits
    rng = np.random.default_rng(3)
    V, N = 6, 5
    parent = np.array([[-1, -1, 0, 0, 2]])
    tokens = np.array([[1, 4, 2, 5, 0]])
    q_row = np.array([[0, 1, 2, 3, 4, 5]])
    for trial in range(40):
        target = rng.normal(0, 1.0, size=(1, N + 1, V))
        draft = rng.normal(0, 1.0, size=(1, N + 1, V))
        ref = verify_tree(target, draft, q_row, tokens, parent, temperature=1.0,
                          draft_kind="logits", seed=trial)
        plen = int(ref.path_len[0])
        path = np.array(ref.path_nodes[0])
        pre = 7
        cache = np.full((1, pre + N, 1), -9)
        cache[0, pre:, 0] = tokens[0]
        nodes = np.full((1, N), -1)
        nodes[0, :plen] = path[:plen]
        out, nl = kv_commit(cache, [pre], [plen], nodes)
        assert nl[0] == pre + plen
        assert list(out[0, pre:pre + plen, 0]) == list(ref.tokens[0][:plen])
