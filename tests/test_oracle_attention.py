"""Pins of the tree-attention oracle (no GPU).

EAGLE-2 notes §4.2: every drafted token sees the committed prefix, its
ancestors and itself.  Pinned against torch's scaled_dot_product_attention
(float64, CPU) with the mask written out position by position, the chain
special case against its causal mask, and invariances the definition fixes.
"""

import numpy as np
import pytest
import torch

from oracle.attention import tree_attention, visible_keys
from oracle.tree import tree_mask


def _inputs(rng, B, N, Hq, Hkv, D, S):
    q = rng.normal(size=(B, N, Hq, D))
    k = rng.normal(size=(B, Hkv, S, D))
    v = rng.normal(size=(B, Hkv, S, D))
    return q, k, v


def _random_parent(rng, B, N):
    return np.array([[-1 if j == 0 or rng.random() < 0.3 else
                      int(rng.integers(0, j)) for j in range(N)]
                     for _ in range(B)])


def _sdpa(q, k, v, prefix, parent, scale):
    """torch SDPA with an explicit boolean mask over [prefix, drafts]."""
    B, N, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    mask, _ = tree_mask(parent)
    out = np.zeros_like(q)
    for b in range(B):
        P = int(prefix[b])
        L = P + N
        allow = np.zeros((N, L), dtype=bool)
        allow[:, :P] = True
        allow[:, P:] = mask[b].astype(bool)
        qb = torch.from_numpy(q[b]).permute(1, 0, 2)             # [Hq, N, D]
        kb = torch.from_numpy(k[b, :, :L]).repeat_interleave(G, 0)
        vb = torch.from_numpy(v[b, :, :L]).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=torch.from_numpy(allow), scale=scale)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_matches_masked_sdpa(Hq, Hkv):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    B, N, D = 3, 9, 16
    prefix = rng.integers(0, 12, size=B)
    S = int(prefix.max()) + N + 2
    q, k, v = _inputs(rng, B, N, Hq, Hkv, D, S)
    parent = _random_parent(rng, B, N)
    scale = 1 / np.sqrt(D)
    got = tree_attention(q, k, v, prefix, parent, scale)
    want = _sdpa(q, k, v, prefix, parent, scale)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_chain_is_causal_attention():
    rng = np.random.default_rng(1)
    B, N, H, D, P = 2, 7, 3, 8, 5
    q, k, v = _inputs(rng, B, N, H, H, D, P + N)
    parent = np.tile(np.arange(-1, N - 1), (B, 1))
    got = tree_attention(q, k, v, [P] * B, parent, 0.5)
    for b in range(B):
        # causal attention of the drafts over [prefix, drafts]
        qb = torch.from_numpy(q[b]).permute(1, 0, 2)
        kb = torch.from_numpy(k[b])
        vb = torch.from_numpy(v[b])
        full_q = torch.zeros(H, P + N, D, dtype=torch.float64)
        full_q[:, P:] = qb
        o = torch.nn.functional.scaled_dot_product_attention(
            full_q, kb, vb, is_causal=True, scale=0.5)
        assert np.allclose(got[b], o[:, P:].permute(1, 0, 2).numpy(),
                           rtol=1e-12, atol=1e-12)


def test_root_child_without_prefix_returns_its_own_value():
    rng = np.random.default_rng(2)
    q, k, v = _inputs(rng, 1, 4, 2, 2, 8, 4)
    parent = np.array([[-1, -1, 0, 1]])
    got = tree_attention(q, k, v, [0], parent, 1.0)
    # node 0 and node 1 see only themselves
    assert np.allclose(got[0, 0], v[0, :, 0])
    assert np.allclose(got[0, 1], v[0, :, 1])


def test_other_branches_do_not_matter():
    rng = np.random.default_rng(3)
    B, N, H, D, P = 1, 8, 2, 8, 6
    q, k, v = _inputs(rng, B, N, H, H, D, P + N)
    parent = np.array([[-1, -1, 0, 0, 1, 2, 2, 4]])
    base = tree_attention(q, k, v, [P], parent, 0.3)
    i = 5                                   # ancestors {0, 2}
    assert visible_keys(parent[0], i, P) == list(range(P)) + [P, P + 2, P + 5]
    k2, v2 = k.copy(), v.copy()
    for j in (1, 3, 4, 6, 7):               # not on node 5's root path
        k2[0, :, P + j] += 5.0
        v2[0, :, P + j] -= 3.0
    moved = tree_attention(q, k2, v2, [P], parent, 0.3)
    assert np.allclose(moved[0, i], base[0, i], rtol=1e-13, atol=1e-13)
    assert not np.allclose(moved[0, 7], base[0, 7])


def test_prefix_order_does_not_matter():
    rng = np.random.default_rng(4)
    B, N, H, D, P = 1, 5, 2, 8, 9
    q, k, v = _inputs(rng, B, N, H, H, D, P + N)
    parent = np.array([[-1, 0, 0, 1, -1]])
    base = tree_attention(q, k, v, [P], parent, 0.4)
    perm = np.concatenate([rng.permutation(P), np.arange(P, P + N)])
    got = tree_attention(q, k[:, :, perm], v[:, :, perm], [P], parent, 0.4)
    assert np.allclose(got, base, rtol=1e-12, atol=1e-12)
