"""Tree attention on the GPU vs the oracle.

Tolerance: the kernel rounds the softmax weights to bf16 before P V (a
relative error of at most 2^-9 per weight, so at most 2^-9 * max|v| on the
output) and rounds the output to bf16 (2^-9 * |o|); accumulation is fp32.
With v ~ N(0, 1) over at most a few thousand keys (max |v| < 5) that is
below 1e-2 + 1e-2 |o|, the bound the tests use.
"""

import numpy as np
import pytest
import torch

import synth
from oracle.attention import tree_attention
from oracle.tree import tree_mask
from tests._parity import lib_ready

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _random_parent(rng, B, N):
    return np.array([[-1 if j == 0 or rng.random() < 0.25 else
                      int(rng.integers(max(0, j - 6), j)) for j in range(N)]
                     for _ in range(B)], dtype=np.int32)


def _bits(parent):
    _, bits = tree_mask(parent)
    return torch.from_numpy(bits.view(np.int64)).cuda()


def _case(seed, B, N, Hq, Hkv, prefix, S, parent=None, D=128):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn(B, N, Hq, D, generator=g, device="cuda").bfloat16()
    k = torch.randn(B, Hkv, S, D, generator=g, device="cuda").bfloat16()
    v = torch.randn(B, Hkv, S, D, generator=g, device="cuda").bfloat16()
    if parent is None:
        parent = _random_parent(np.random.default_rng(seed), B, N)
    pre = torch.tensor(prefix, dtype=torch.int32, device="cuda")
    return q, k, v, pre, parent


def _check(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), float(err.max())


@pytest.mark.parametrize("N,Hq,Hkv,prefix", [
    (1, 4, 4, [0, 5]),
    (7, 8, 2, [1, 63]),
    (16, 4, 1, [64, 65]),          # prefix ends exactly on a tile
    (60, 32, 8, [130, 0]),         # the static-tree shape, tree-only sequence
    (64, 2, 2, [200, 191]),        # 64 drafted nodes (full mask word)
    (33, 6, 3, [127, 129]),        # 66 rows: a second, ragged CTA
])
def test_tree_attention_matches_oracle(N, Hq, Hkv, prefix):
    B = len(prefix)
    S = max(prefix) + N + 9
    q, k, v, pre, parent = _case(N * 100 + Hq, B, N, Hq, Hkv, prefix, S)
    out = api().spec_tree_attention(q, k, v, pre, _bits(parent),
                                    scale=128 ** -0.5)
    torch.cuda.synchronize()
    ref = tree_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                         v.float().cpu().numpy(), prefix, parent,
                         128 ** -0.5)
    _check(out, ref)


def test_many_sequences_longest_first_with_ties():
    # the CTAs take sequences longest first (ties by index): every sequence,
    # equal prefixes included, must still land in its own output rows
    prefix = [5, 300, 300, 0, 129, 64, 300, 1, 257, 5, 77, 200]
    B, N, Hq, Hkv = len(prefix), 7, 8, 2
    S = max(prefix) + N + 3
    q, k, v, pre, parent = _case(31, B, N, Hq, Hkv, prefix, S)
    out = api().spec_tree_attention(q, k, v, pre, _bits(parent), scale=0.09)
    torch.cuda.synchronize()
    ref = tree_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                         v.float().cpu().numpy(), prefix, parent, 0.09)
    _check(out, ref)


def test_chain_and_static_tree_masks():
    w = synth.workload("tree_static")
    static = synth.static_tree(w).numpy()
    N = static.size
    chain = np.arange(-1, N - 1, dtype=np.int32)
    parent = np.stack([static, chain, static])
    prefix = [300, 77, 0]
    q, k, v, pre, _ = _case(7, 3, N, 8, 2, prefix, 400 + N, parent)
    out = api().spec_tree_attention(q, k, v, pre, _bits(parent), scale=0.05)
    torch.cuda.synchronize()
    ref = tree_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                         v.float().cpu().numpy(), prefix, parent, 0.05)
    _check(out, ref)


def test_prefix_is_clamped_to_the_cache():
    # a prefix longer than S - N reads the last S - N positions as prefix
    N, S = 5, 40
    q, k, v, pre, parent = _case(9, 1, N, 2, 2, [1000], S)
    out = api().spec_tree_attention(q, k, v, pre, _bits(parent), scale=0.1)
    torch.cuda.synchronize()
    ref = tree_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                         v.float().cpu().numpy(), [S - N], parent, 0.1)
    _check(out, ref)


def test_full_size_sampled_sequences():
    # the bench workload: B = 32, 60-node static tree, 32 query heads over
    # 8 key/value heads, head dim 128, prefixes 2048..4095; two sequences
    # checked against the oracle in full
    rng = np.random.default_rng(21)
    B, Hq, Hkv, S = 32, 32, 8, 4096 + 64
    w = synth.workload("tree_static")
    static = synth.static_tree(w).numpy()
    N = static.size
    parent = np.tile(static, (B, 1))
    prefix = rng.integers(2048, 4096, size=B).astype(np.int32)
    q, k, v, pre, _ = _case(23, B, N, Hq, Hkv, list(prefix), S, parent)
    out = api().spec_tree_attention(q, k, v, pre, _bits(parent))
    torch.cuda.synchronize()
    for b in (0, 17):
        ref = tree_attention(q[b:b + 1].float().cpu().numpy(),
                             k[b:b + 1].float().cpu().numpy(),
                             v[b:b + 1].float().cpu().numpy(), prefix[b:b + 1],
                             parent[b:b + 1], 128 ** -0.5)
        _check(out[b:b + 1], ref)
    assert torch.isfinite(out.float()).all()
