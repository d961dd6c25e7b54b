"""Sampled chain verification (full vocabulary) vs the oracle.

Accept / reject decisions, replacement and bonus tokens must be bit-exact
except on sequences where a uniform lies within 1e-5 of its threshold or CDF
boundary (the oracle flags those); the acceptance mass agrees to rel 1e-4."""

import numpy as np
import pytest
import torch

import synth
from oracle.chain import verify_chain
from tests._parity import compare_chain, lib_ready, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def run(w, seqs=None, target=None, draft=None, toks=None, seed=None):
    if target is None:
        target, draft, toks = synth.chain_inputs(w, "cuda")
    seed = w.decision_seed if seed is None else seed
    gpu = api().spec_verify_chain(target, draft, toks,
                                  temperature=w.temperature, top_k=w.top_k,
                                  top_p=w.top_p, draft_kind=w.draft_kind,
                                  seed=seed)
    torch.cuda.synchronize()
    sel = slice(None) if seqs is None else seqs
    ref = verify_chain(np64(target[sel]), np64(draft[sel]),
                       toks[sel].cpu().numpy(), temperature=w.temperature,
                       top_k=w.top_k, top_p=w.top_p,
                       draft_kind=w.draft_kind, seed=seed,
                       batch_ids=None if seqs is None else seqs)
    return gpu, ref


def test_chain_sample_workload_exact():
    # B=1, K=4, V=32000 float32, the pages' alpha ~ 0.8 chain
    w = synth.workload("chain_sample")
    for seed in range(1, 41):
        gpu, ref = run(w, seed=seed)
        compare_chain(gpu, ref)


@pytest.mark.parametrize("V", [1, 2, 37, 1000, 4099, 32000, 70001])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_chain_vocab_sizes(V, dt):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    w = synth.workload("chain_sample", B=6, K=3, V=V, target_dtype=tdt,
                       draft_dtype=tdt, seed=77 + V)
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)


@pytest.mark.parametrize("V,dt", [(300000, "bf16"), (150001, "f32")])
def test_chain_large_vocab(V, dt):
    # V = 300000 (aligned): the streaming kernel with 4-CTA clusters;
    # V = 150001 (odd row length): the general kernel, 8-CTA clusters
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    w = synth.workload("chain_sample", B=3, K=2, V=V, target_dtype=tdt,
                       draft_dtype=tdt, seed=V % 1000)
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_chain_probs_draft(T):
    w = synth.workload("chain_sample", B=8, K=4, V=5000, draft_kind="probs",
                       temperature=T, seed=5)
    gpu, ref = run(w)
    compare_chain(gpu, ref)


def test_chain_mixed_dtypes_and_low_alpha():
    w = synth.workload("chain_sample", B=16, K=6, V=20000,
                       target_dtype=torch.bfloat16, draft_dtype=torch.float32,
                       draft_noise=3.0, seed=9)
    gpu, ref = run(w)
    compare_chain(gpu, ref)
    assert (ref.accepted < 6).any()


def test_chain_identical_rows_accept_all_and_bonus():
    w = synth.workload("chain_sample", B=4, K=3, V=3000, seed=2)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    draft = target[:, :3].contiguous()
    gpu, ref = run(w, target=target, draft=draft, toks=toks)
    compare_chain(gpu, ref)
    assert (gpu[0].cpu() == 3).all()
    np.testing.assert_allclose(gpu[2].cpu().numpy(), 1.0, rtol=1e-5)


def test_chain_zero_q_and_out_of_range_tokens():
    from speculative_decoding_verification_tree_gb300 import _lib
    V = 700
    w = synth.workload("chain_sample", B=3, K=2, V=V, seed=3)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    draft[0, 0, 11] = float("-inf")
    toks[0, 0] = 11             # q(x) = 0: accepted
    toks[1, 1] = V + 5          # out of range: rejected
    toks[2, 0] = -1
    a = api()
    ws = a.workspace(_lib.SPEC_OP_CHAIN, 3, 2, V)
    gpu = a.spec_verify_chain(target, draft, toks, temperature=1.0,
                              seed=w.decision_seed, ws=ws)
    st = a.spec_get_status(ws)
    ref = verify_chain(np64(target), np64(draft), toks.cpu().numpy(),
                       temperature=1.0, seed=w.decision_seed)
    compare_chain(gpu, ref)
    assert st & _lib.SPEC_STATUS_QZERO_ACCEPT
    assert st & _lib.SPEC_STATUS_TOKEN_RANGE
    assert st == ref.status


def test_chain_batched_full_vocab_llama_size():
    # many sequences at V = 128256, compared on a sample of sequences
    w = synth.workload("chain_sample", B=48, K=5, V=128256,
                       target_dtype=torch.bfloat16,
                       draft_dtype=torch.bfloat16, seed=11)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    seqs = list(range(w.B))  # all 48 sequences
    gpu, ref = run(w, seqs=seqs, target=target, draft=draft, toks=toks)
    p = compare_chain(gpu, ref, seqs=seqs, max_excluded=2)
    assert p.exact >= w.B - 4, p


# ---- the single-launch form: a few sampled chains with every row resident
# in shared memory (one cluster of 8 CTAs per sequence)

@pytest.mark.parametrize("V", [8, 16, 24, 64, 4096, 32000])
def test_chain_small_vocab_slices(V):
    # V = 8..24: some of the 8 CTAs own no part of the vocabulary
    w = synth.workload("chain_sample", B=5, K=3, V=V, seed=500 + V)
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)


@pytest.mark.parametrize("B", [19, 20])
def test_chain_small_longest_chain_and_wave_edge(B):
    # K = 16 drafts (the most the single launch takes); B = 19 fills one wave
    # of 8-CTA clusters on 152 SMs, B = 20 goes to the streaming kernel
    w = synth.workload("chain_sample", B=B, K=16, V=4096,
                       target_dtype=torch.bfloat16,
                       draft_dtype=torch.bfloat16, draft_noise=0.3, seed=B)
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)
    assert (ref.accepted > 4).any()


@pytest.mark.parametrize("T", [1.0, 0.6])
@pytest.mark.parametrize("ddt", [torch.float32, torch.bfloat16])
def test_chain_small_probs_draft(T, ddt):
    w = synth.workload("chain_sample", B=4, K=5, V=12000, draft_kind="probs",
                       draft_dtype=ddt, temperature=T, seed=int(T * 10))
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)


def test_chain_small_zero_q_and_out_of_range_tokens():
    from speculative_decoding_verification_tree_gb300 import _lib
    V = 704
    w = synth.workload("chain_sample", B=3, K=2, V=V, seed=4)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    draft[0, 0, 11] = float("-inf")
    toks[0, 0] = 11             # q(x) = 0: accepted
    toks[1, 1] = V + 5          # out of range: rejected
    toks[2, 0] = -1
    a = api()
    ws = a.workspace(_lib.SPEC_OP_CHAIN, 3, 2, V)
    gpu = a.spec_verify_chain(target, draft, toks, temperature=1.0,
                              seed=w.decision_seed, ws=ws)
    st = a.spec_get_status(ws)
    ref = verify_chain(np64(target), np64(draft), toks.cpu().numpy(),
                       temperature=1.0, seed=w.decision_seed)
    compare_chain(gpu, ref)
    assert st & _lib.SPEC_STATUS_QZERO_ACCEPT
    assert st & _lib.SPEC_STATUS_TOKEN_RANGE
    assert st == ref.status


def test_chain_small_bonus_from_p_when_all_accepted():
    # draft == target: every token accepted, the bonus drawn from p_K
    w = synth.workload("chain_sample", B=6, K=4, V=2048, seed=6)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    draft = target[:, :4].contiguous()
    gpu, ref = run(w, target=target, draft=draft, toks=toks)
    compare_chain(gpu, ref)
    assert (gpu[0].cpu() == 4).all()
    np.testing.assert_allclose(gpu[2].cpu().numpy(), 1.0, rtol=1e-5)


def test_chain_small_single_sequence_rewrites_status():
    # one sequence: the single cluster writes the whole status word, so a
    # flag of the previous call on the same workspace must not survive
    from speculative_decoding_verification_tree_gb300 import _lib
    V = 704
    w = synth.workload("chain_sample", B=1, K=2, V=V, seed=8)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    a = api()
    ws = a.workspace(_lib.SPEC_OP_CHAIN, 1, 2, V)
    bad = toks.clone()
    bad[0, 0] = V + 1            # out of range: rejected, flagged
    gpu = a.spec_verify_chain(target, draft, bad, temperature=1.0,
                              seed=w.decision_seed, ws=ws)
    assert a.spec_get_status(ws) & _lib.SPEC_STATUS_TOKEN_RANGE
    ref = verify_chain(np64(target), np64(draft), bad.cpu().numpy(),
                       temperature=1.0, seed=w.decision_seed)
    compare_chain(gpu, ref)
    gpu = a.spec_verify_chain(target, draft, toks, temperature=1.0,
                              seed=w.decision_seed, ws=ws)
    st = a.spec_get_status(ws)
    ref = verify_chain(np64(target), np64(draft), toks.cpu().numpy(),
                       temperature=1.0, seed=w.decision_seed)
    compare_chain(gpu, ref)
    assert st == ref.status == 0


@pytest.mark.parametrize("K", [2, 3])
def test_chain_small_shared_memory_limit_llama_vocab(K):
    # V = 128256 bf16: K = 2 keeps five 32 KB row slices per CTA (160 KB,
    # the single launch); K = 3 needs seven (224 KB) and streams instead
    w = synth.workload("chain_sample", B=2, K=K, V=128256,
                       target_dtype=torch.bfloat16,
                       draft_dtype=torch.bfloat16, seed=40 + K)
    gpu, ref = run(w)
    compare_chain(gpu, ref, max_excluded=1)
