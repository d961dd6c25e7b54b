"""KV-cache commit on the GPU vs the oracle (bit-exact bytes)."""

import numpy as np
import pytest
import torch

from oracle.kv import kv_commit
from tests._parity import lib_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _paths(rng, B, N, invalid=()):
    """Random strictly increasing paths (tree paths are node subsequences)."""
    lens = rng.integers(0, N + 1, size=B).astype(np.int32)
    nodes = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        nodes[b, :lens[b]] = np.sort(rng.choice(N, size=lens[b], replace=False))
    for b in invalid:  # out of order or out of range
        if lens[b] >= 2:
            nodes[b, 0], nodes[b, 1] = nodes[b, 1], nodes[b, 0]
        else:
            lens[b] = N + 1
    return lens, nodes


def _bits(t):
    """Raw element bits of a tensor as numpy (bf16 -> int16)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.cpu().numpy()


def _run(cache, layout, row_bytes, pre, lens, nodes, N):
    dev = cache.device
    p = torch.tensor(pre, dtype=torch.int32, device=dev)
    l = torch.tensor(lens, dtype=torch.int32, device=dev)
    nd = None if nodes is None else torch.tensor(nodes, dtype=torch.int32,
                                                 device=dev)
    nl = api().spec_kv_commit(cache, p, l, nd, layout=layout,
                              row_bytes=row_bytes, N=N)
    torch.cuda.synchronize()
    return nl.cpu().numpy()


def test_head_major_bf16_16_byte_rows():
    rng = np.random.default_rng(0)
    n1, B, n2, D, N = 4, 5, 3, 64, 9
    pre = rng.integers(0, 20, size=B).astype(np.int32)
    S = int(pre.max()) + N + 3
    cache = torch.randn(n1, B, n2, S, D, dtype=torch.bfloat16, device="cuda")
    es = 2
    layout = (n1, n2, n2 * S * D * es, B * n2 * S * D * es, S * D * es, D * es)
    lens, nodes = _paths(rng, B, N, invalid=[3])
    before = _bits(cache).transpose(1, 3, 0, 2, 4)       # [B, S, n1, n2, D]
    nl = _run(cache, layout, D * es, pre, lens, nodes, N)
    ref, ref_len = kv_commit(before, pre, lens, nodes)
    assert np.array_equal(nl, ref_len)
    assert nl[3] == -1
    assert np.array_equal(_bits(cache).transpose(1, 3, 0, 2, 4), ref)


@pytest.mark.parametrize("dtype,W", [(torch.float32, 7), (torch.uint8, 5)])
def test_position_major_narrow_rows(dtype, W):
    # 28-byte rows take the 4-byte copy, 5-byte rows the byte copy
    rng = np.random.default_rng(W)
    B, N = 6, 12
    pre = rng.integers(0, 30, size=B).astype(np.int32)
    S = int(pre.max()) + N
    if dtype == torch.uint8:
        cache = torch.randint(0, 256, (B, S, W), dtype=dtype, device="cuda")
    else:
        cache = torch.randn(B, S, W, dtype=dtype, device="cuda")
    es = cache.element_size()
    layout = (1, 1, S * W * es, 0, 0, W * es)
    lens, nodes = _paths(rng, B, N)
    before = cache.cpu().numpy()
    nl = _run(cache, layout, W * es, pre, lens, nodes, N)
    ref, ref_len = kv_commit(before, pre, lens, nodes)
    assert np.array_equal(nl, ref_len)
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_chain_moves_nothing_and_sets_lengths():
    B, K = 4, 5
    cache = torch.randn(B, 40, 8, device="cuda")
    before = cache.clone()
    pre = np.array([3, 0, 17, 30], dtype=np.int32)
    acc = np.array([0, 5, 2, 6], dtype=np.int32)  # 6 > K: refused
    nl = _run(cache, (1, 1, 40 * 32, 0, 0, 32), 32, pre, acc, None, K)
    assert list(nl) == [3, 5, 19, -1]
    assert torch.equal(cache, before)


def test_empty_batch_and_identity_paths():
    a = api()
    z = torch.empty(0, dtype=torch.int32, device="cuda")
    out = a.spec_kv_commit(torch.empty(0, device="cuda"), z, z, None,
                           layout=(1, 1, 0, 0, 0, 16), row_bytes=16, N=4)
    assert out.numel() == 0
    cache = torch.randn(2, 16, 4, device="cuda")
    before = cache.clone()
    nodes = np.array([[0, 1, 2, -1], [0, 1, 2, 3]], dtype=np.int32)
    nl = _run(cache, (1, 1, 16 * 16, 0, 0, 16), 16, np.array([2, 5]),
              np.array([3, 4]), nodes, 4)
    assert list(nl) == [5, 9]
    assert torch.equal(cache, before)


def test_model_sized_cache_sampled_planes():
    # 32 layers x (K, V) x 8 KV heads x 128 dims bf16, head-major, B = 32,
    # 60-node paths (the static tree's sizes), prefixes up to 200 positions
    rng = np.random.default_rng(7)
    n1, B, n2, D, N = 64, 32, 8, 128, 60
    pre = rng.integers(0, 200, size=B).astype(np.int32)
    S = int(pre.max()) + N
    cache = torch.randn(n1, B, n2, S, D, dtype=torch.bfloat16, device="cuda")
    es = 2
    layout = (n1, n2, n2 * S * D * es, B * n2 * S * D * es, S * D * es, D * es)
    lens = rng.integers(0, 7, size=B).astype(np.int32)
    nodes = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        nodes[b, :lens[b]] = np.sort(rng.choice(N, size=lens[b], replace=False))
    planes = [(0, 0), (0, 7), (37, 3), (63, 7)]
    before = {pl: _bits(cache[pl[0], :, pl[1]]) for pl in planes}  # [B, S, D]
    nl = _run(cache, layout, D * es, pre, lens, nodes, N)
    for pl in planes:
        ref, ref_len = kv_commit(before[pl], pre, lens, nodes)
        assert np.array_equal(_bits(cache[pl[0], :, pl[1]]), ref), pl
    assert np.array_equal(nl, ref_len)
