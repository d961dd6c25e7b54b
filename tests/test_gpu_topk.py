"""Sampled verification with top-k / top-p truncation vs the oracle.

The transform (temperature, then top-k with ties to the lower index, then
top-p over the kept tokens, each followed by renormalisation) is applied to
target and draft alike.  Top-k membership is exact; decisions and tokens are
exact except on sequences where an accept test or a top-p cut lies within
1e-5 of its threshold (excluded and counted), and replacement / bonus draws
may only differ within the 1e-5 band of a CDF boundary."""

import numpy as np
import pytest
import torch

import synth
from oracle.chain import verify_chain
from oracle.tree import verify_tree
from tests._parity import compare_chain, compare_tree, lib_ready, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def run_chain(w, target=None, draft=None, toks=None, seed=None):
    if target is None:
        target, draft, toks = synth.chain_inputs(w, "cuda")
    seed = w.decision_seed if seed is None else seed
    gpu = api().spec_verify_chain(target, draft, toks,
                                  temperature=w.temperature, top_k=w.top_k,
                                  top_p=w.top_p, draft_kind=w.draft_kind,
                                  seed=seed)
    torch.cuda.synchronize()
    ref = verify_chain(np64(target), np64(draft), toks.cpu().numpy(),
                       temperature=w.temperature, top_k=w.top_k,
                       top_p=w.top_p, draft_kind=w.draft_kind, seed=seed)
    return gpu, ref


def test_topk_topp_workload_full():
    # B=64, K=5, V=32000 bf16, T=0.7, top-k 50, top-p 0.9 on both sides
    w = synth.workload("chain_topk")
    gpu, ref = run_chain(w)
    compare_chain(gpu, ref, max_excluded=3)
    assert ref.status == 0


@pytest.mark.parametrize("k,p", [(1, 1.0), (5, 1.0), (50, 0.5), (128, 0.95),
                                 (128, 1.0), (7, 0.3)])
def test_topk_variants(k, p):
    w = synth.workload("chain_topk", B=24, K=3, V=3001, top_k=k, top_p=p,
                       seed=k * 10 + int(p * 10))
    gpu, ref = run_chain(w)
    compare_chain(gpu, ref, max_excluded=2)


def test_topp_only_small_vocab():
    w = synth.workload("chain_topk", B=16, K=4, V=100, top_k=0, top_p=0.8,
                       seed=3)
    gpu, ref = run_chain(w)
    compare_chain(gpu, ref)


def test_topk_exact_ties_and_fp32_probs():
    # integer logits: many exact ties at the k-th value (lower index wins)
    B, K, V = 12, 3, 2000
    g = torch.Generator(device="cpu").manual_seed(9)
    t = torch.randint(-4, 4, (B, K + 1, V), generator=g).float()
    d = t[:, :K] + torch.randint(-1, 2, (B, K, V), generator=g).float()
    # top_p 0.83 lies between the cumulative sums of the 20 equal kept
    # probabilities (0.05 each), so the cut itself is no near tie
    w = synth.workload("chain_topk", B=B, K=K, V=V, top_k=20, top_p=0.83,
                       temperature=1.3, seed=1)
    target = t.to(torch.bfloat16).cuda()
    draft = d.to(torch.bfloat16).cuda()
    toks = torch.randint(0, V, (B, K), generator=g).to(torch.int32).cuda()
    # make half the drafted tokens come from the kept set
    am = torch.argmax(d, -1).to(torch.int32).cuda()
    toks[:, ::2] = am[:, ::2]
    gpu, ref = run_chain(w, target, draft, toks)
    compare_chain(gpu, ref)
    # probabilities as draft rows (float32)
    w2 = synth.workload("chain_topk", B=B, K=K, V=V, top_k=20, top_p=1.0,
                        draft_kind="probs", draft_dtype=torch.float32,
                        seed=1)
    probs = torch.softmax(d, -1).cuda()
    gpu, ref = run_chain(w2, target, probs, toks)
    compare_chain(gpu, ref)


def test_topk_tree():
    w = synth.workload("tree_static", B=6, V=4000, top_k=16, top_p=0.9,
                       draft_kind="logits", draft_dtype=torch.bfloat16,
                       temperature=0.8, seed=12)
    target, draft, q_row, toks, par = synth.tree_inputs(w, "cuda")
    gpu = api().spec_verify_tree(target, draft, q_row, toks, par,
                                 temperature=w.temperature, top_k=w.top_k,
                                 top_p=w.top_p, seed=w.decision_seed)
    torch.cuda.synchronize()
    ref = verify_tree(np64(target), np64(draft), q_row.cpu().numpy(),
                      toks.cpu().numpy(), par.cpu().numpy(),
                      temperature=w.temperature, top_k=w.top_k, top_p=w.top_p,
                      seed=w.decision_seed)
    compare_tree(gpu, ref, max_excluded=1)


@pytest.mark.parametrize("V,dt", [(128256, torch.bfloat16),
                                  (90000, torch.float32)])
def test_topk_long_rows_rescan_flagged_threads(V, dt):
    # rows of more groups per thread than the group-key table holds: the
    # threads whose maximum reaches the bound rescan all their groups
    w = synth.workload("chain_topk", B=4, K=3, V=V, target_dtype=dt,
                       draft_dtype=dt, seed=V % 977)
    gpu, ref = run_chain(w)
    compare_chain(gpu, ref, max_excluded=1)


def test_topk_constant_rows_overflow_the_candidates():
    # every logit of a row ties at the bound: more candidates than the
    # shared list holds, so the row takes the exact fallback selection (the
    # k lowest indices of the tied value)
    w = synth.workload("chain_topk", B=3, K=2, V=32000, top_k=50, top_p=1.0,
                       seed=17)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    target[0].zero_()
    draft[1].fill_(1.5)
    toks[0, 0] = 7        # inside the tied row's top-k
    toks[1, 1] = 40000 % w.V
    gpu, ref = run_chain(w, target=target, draft=draft, toks=toks)
    compare_chain(gpu, ref, max_excluded=1)
