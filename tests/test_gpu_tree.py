"""Tree attention mask, tree verification and the Philox generator vs the
oracle."""

import numpy as np
import pytest
import torch

import synth
from oracle import philox
from oracle.tree import tree_mask, verify_tree
from tests._parity import compare_tree, lib_ready, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _random_parents(B, N, seed, max_kids=None):
    rng = np.random.default_rng(seed)
    par = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        kids = {}
        for j in range(N):
            while True:
                p = int(rng.integers(-1, j)) if j else -1
                if max_kids is None or kids.get(p, 0) < max_kids:
                    break
            kids[p] = kids.get(p, 0) + 1
            par[b, j] = p
    return par


@pytest.mark.parametrize("N", [1, 5, 60, 64, 65, 300])
def test_tree_mask_random(N):
    par = _random_parents(5, N, N)
    pt = torch.from_numpy(par).cuda()
    m, bits = api().spec_tree_mask(pt, bits=N <= 64)
    want, wbits = tree_mask(par)
    assert np.array_equal(m.cpu().numpy(), want)
    if N <= 64:
        assert np.array_equal(bits.cpu().numpy().view(np.uint64), wbits)


def test_tree_mask_static_and_chain():
    w = synth.workload("tree_static")
    par = synth.static_tree(w).reshape(1, -1).repeat(3, 1)
    m, bits = api().spec_tree_mask(par.cuda(), bits=True)
    want, wbits = tree_mask(par.numpy())
    assert np.array_equal(m.cpu().numpy(), want)
    assert np.array_equal(bits.cpu().numpy().view(np.uint64), wbits)
    chain = torch.arange(-1, 9, dtype=torch.int32).reshape(1, 10).cuda()
    m, _ = api().spec_tree_mask(chain)
    assert np.array_equal(m[0].cpu().numpy(), np.tril(np.ones((10, 10))))


def test_tree_mask_invalid_parent_stops_walk():
    par = np.array([[-1, 0, 5, 1, -7]], dtype=np.int32)
    m, _ = api().spec_tree_mask(torch.from_numpy(par).cuda())
    want, _ = tree_mask(par)
    assert np.array_equal(m.cpu().numpy(), want)


def test_philox_bit_exact():
    rng = np.random.default_rng(0)
    n = 4096
    b = rng.integers(0, 1 << 31, n).astype(np.int32)
    i = rng.integers(0, 1 << 31, n).astype(np.int32)
    s = rng.integers(0, 2, n).astype(np.int32)
    for seed, off in [(0, 0), (1, 0), (2**40 + 17, 3), (2**64 - 1, 2**32 - 1)]:
        out = api().spec_philox_uniforms(
            seed, off, torch.from_numpy(b).cuda(), torch.from_numpy(i).cuda(),
            torch.from_numpy(s).cuda()).cpu().numpy()
        want = philox.uniform_np(seed, b.astype(np.uint64),
                                 i.astype(np.uint64), s.astype(np.uint64),
                                 off)
        assert np.array_equal(out.astype(np.float64), want)


def run_tree(w, target, draft, q_row, toks, par, seqs=None, seed=None):
    seed = w.decision_seed if seed is None else seed
    gpu = api().spec_verify_tree(target, draft, q_row, toks, par,
                                 temperature=w.temperature, top_k=w.top_k,
                                 top_p=w.top_p, draft_kind=w.draft_kind,
                                 seed=seed)
    torch.cuda.synchronize()
    sel = slice(None) if seqs is None else seqs
    ref = verify_tree(np64(target[sel]), np64(draft[sel]),
                      q_row[sel].cpu().numpy(), toks[sel].cpu().numpy(),
                      par[sel].cpu().numpy(), temperature=w.temperature,
                      top_k=w.top_k, top_p=w.top_p, draft_kind=w.draft_kind,
                      seed=seed, batch_ids=None if seqs is None else seqs)
    return gpu, ref


@pytest.mark.parametrize("V", [3, 1000, 9001])
def test_static_tree_small_vocab(V):
    w = synth.workload("tree_static", B=8, V=V, seed=40 + V)
    ins = synth.tree_inputs(w, "cuda")
    gpu, ref = run_tree(w, *ins)
    compare_tree(gpu, ref, max_excluded=1)


def test_static_tree_large_vocab():
    # aligned V = 300000: 4-CTA clusters in the streaming kernel and the walk
    w = synth.workload("tree_static", B=2, V=300000, seed=8)
    ins = synth.tree_inputs(w, "cuda")
    gpu, ref = run_tree(w, *ins)
    compare_tree(gpu, ref, max_excluded=1)


def test_static_tree_low_acceptance_many_sibling_passes():
    # noisy draft: most first children are rejected, siblings are tried
    w = synth.workload("tree_static", B=12, V=2000, draft_noise=3.0, seed=5)
    ins = synth.tree_inputs(w, "cuda")
    for seed in (1, 2, 3):
        gpu, ref = run_tree(w, *ins, seed=seed)
        compare_tree(gpu, ref)


def test_random_trees_logits_draft():
    B, N, V = 6, 40, 1500
    par = torch.from_numpy(_random_parents(B, N, 9, max_kids=6)).cuda()
    w = synth.workload("tree_static", B=B, V=V, draft_kind="logits",
                       draft_dtype=torch.bfloat16, temperature=0.9, seed=3)
    # per-sequence parents: build the tree inputs with sequence 0's parents,
    # then use each sequence's own parents (tokens are drawn per row anyway)
    target, draft, q_row, toks, _ = synth.tree_inputs(w, "cuda", par[0])
    gpu, ref = run_tree(w, target, draft, q_row, toks, par)
    compare_tree(gpu, ref)


def test_tree_partial_draft_rows():
    # only rows with children carry a draft row (q_row = -1 elsewhere)
    w = synth.workload("tree_static", B=5, V=2500, seed=8)
    target, draft, q_row, toks, par = synth.tree_inputs(w, "cuda")
    haskid = np.zeros(61, dtype=bool)
    for p in par[0].tolist():
        haskid[p + 1] = True
    q_row[:, ~torch.from_numpy(haskid).cuda()] = -1
    gpu, ref = run_tree(w, target, draft, q_row, toks, par)
    compare_tree(gpu, ref)


def test_static_tree_full_size_sampled():
    # B=32, 60 nodes, V=128256, bf16 target + float32 draft probabilities
    w = synth.workload("tree_static")
    ins = synth.tree_inputs(w, "cuda")
    # every sequence of the batch against the oracle (about 40 s of CPU)
    seqs = list(range(w.B))
    gpu, ref = run_tree(w, *ins, seqs=seqs)
    p = compare_tree(gpu, ref, seqs=seqs, max_excluded=2)
    assert p.exact >= w.B - 4, p
