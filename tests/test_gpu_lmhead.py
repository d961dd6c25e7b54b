"""GPU parity of the target LM head (spec_lm_head) and of tree verification
through it (spec_verify_tree_lmhead) against the oracle (oracle/lmhead.py).

Logits: every bf16 logit lies in the oracle's range [RN(z - delta),
RN(z + delta)] of the exact product z, delta the float32 accumulation bound
(a single value, the nearest rounding, except near rounding midpoints and
near zero).  Row normalisers:
within 2e-5 of the oracle's on its rounded logits (a handful of ambiguous
logits may round the other way, each moving the normaliser by under 1e-6).
Verification: the rules of the other tree tests, with rounding near ties
(the two roundings decide a sequence differently) counted with the accept
near ties.
"""

import numpy as np
import pytest
import torch

import synth
from oracle.lmhead import lm_head_logits, verify_tree_lmhead
from tests._parity import compare_tree, lib_ready, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _inputs(M, H, V, seed, std=2.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w = (torch.randn(V, H, generator=g, device="cuda") * (std / H ** 0.5)) \
        .bfloat16()
    return h, w


def _check_logits(got, lg):
    """got: GPU logits (float64 numpy) of the rows lg covers.  Returns how
    many differ from the nearest rounding (all of them ambiguous)."""
    bad = ~((lg.lo <= got) & (got <= lg.hi))
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:5].tolist())
    return int((got != lg.rn).sum())


@pytest.mark.parametrize("M,H,V", [(1, 64, 256), (128, 64, 256),
                                   (200, 192, 1000), (130, 512, 4099),
                                   (257, 136, 777)])
def test_lm_head_logits_and_normalisers(M, H, V):
    h, w = _inputs(M, H, V, seed=M + H + V)
    T = 0.8
    logits, lse = api().spec_lm_head(h, w, temperature=T, row_lse=True)
    torch.cuda.synchronize()
    lg = lm_head_logits(np64(h), np64(w))
    _check_logits(np64(logits), lg)
    kt = np.log2(np.e) / T
    want = np.log2(np.exp2(lg.rn * kt - (lg.rn * kt).max(-1, keepdims=True))
                   .sum(-1)) + (lg.rn * kt).max(-1)
    np.testing.assert_allclose(lse.cpu().numpy(), want, rtol=2e-5, atol=2e-5)


def test_lm_head_full_vocab_sampled_rows():
    # the static-tree batch's shape: 1952 rows x H 4096 x V 128256; rows from
    # the first, a middle and the ragged last 128-row tile, checked in full
    M, H, V = 32 * 61, 4096, 128256
    h, w = _inputs(M, H, V, seed=7)
    logits, lse = api().spec_lm_head(h, w, temperature=1.0, row_lse=True)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 1000, 1919, 1920, M - 1]
    lg = lm_head_logits(np64(h[rows]), np64(w))
    flips = _check_logits(np64(logits[rows]), lg)
    assert flips <= 0.01 * len(rows) * V
    kt = np.log2(np.e)
    z = lg.rn * kt
    want = np.log2(np.exp2(z - z.max(-1, keepdims=True)).sum(-1)) + z.max(-1)
    np.testing.assert_allclose(lse[rows].cpu().numpy(), want, rtol=2e-5,
                               atol=2e-5)


def test_lm_head_status_and_determinism():
    from speculative_decoding_verification_tree_gb300 import _lib
    M, H, V = 300, 256, 5000
    h, w = _inputs(M, H, V, seed=3)
    ws = api().workspace(_lib.SPEC_OP_LMHEAD, M, 0, V)
    a, la = api().spec_lm_head(h, w, temperature=0.7, row_lse=True, ws=ws)
    assert api().spec_get_status(ws) == 0
    b, lb = api().spec_lm_head(h, w, temperature=0.7, row_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


def _run_tree(w, ins, seqs):
    hidden, wv, draft, q_row, toks, par = ins
    logits = torch.empty(hidden.shape[0], hidden.shape[1], wv.shape[0],
                         dtype=torch.bfloat16, device="cuda")
    from speculative_decoding_verification_tree_gb300 import _lib
    ws = api().workspace(_lib.SPEC_OP_TREE_LMHEAD, w.B, toks.shape[1], w.V)
    gpu = api().spec_verify_tree_lmhead(
        hidden, wv, draft, q_row, toks, par, temperature=w.temperature,
        draft_kind=w.draft_kind, seed=w.decision_seed, logits=logits, ws=ws)
    torch.cuda.synchronize()
    assert api().spec_get_status(ws) == 0
    res = verify_tree_lmhead(
        np64(hidden[seqs]), np64(wv), np64(draft[seqs]),
        q_row[seqs].cpu().numpy(), toks[seqs].cpu().numpy(),
        par[seqs].cpu().numpy(), temperature=w.temperature,
        draft_kind=w.draft_kind, seed=w.decision_seed, batch_ids=seqs)
    _check_logits(np64(logits[seqs]), res.logits)
    return gpu, res


@pytest.mark.parametrize("V,H,B", [(4099, 256, 4), (32000, 1024, 3)])
def test_tree_lmhead_small(V, H, B):
    w = synth.workload("lmhead_tree", B=B, V=V, H=H, seed=V + H)
    ins = synth.lmhead_tree_inputs(w, "cuda")
    seqs = list(range(B))
    gpu, res = _run_tree(w, ins, seqs)
    compare_tree(gpu, res.ref, seqs=seqs, max_excluded=1,
                 mass_slack=res.mass_slack)


def test_tree_lmhead_greedy():
    w = synth.workload("lmhead_tree", B=3, V=3000, H=128, temperature=0.0,
                       seed=5)
    ins = synth.lmhead_tree_inputs(
        synth.workload("lmhead_tree", B=3, V=3000, H=128, seed=5), "cuda")
    # the draft rows and q_row are passed but not read at temperature 0
    seqs = [0, 1, 2]
    gpu, res = _run_tree(w, ins, seqs)
    compare_tree(gpu, res.ref, greedy=True, seqs=seqs, max_excluded=1)


def test_tree_lmhead_full_size_sampled():
    # B = 32, 60 nodes, V = 128256, H = 4096: the GEMM over all 1952 rows,
    # eight sequences checked against the oracle one by one
    w = synth.workload("lmhead_tree")
    ins = synth.lmhead_tree_inputs(w, "cuda")
    seqs = [0, 5, 11, 17, 22, 26, 30, 31]
    gpu, res = _run_tree(w, ins, seqs)
    p = compare_tree(gpu, res.ref, seqs=seqs, max_excluded=2,
                     mass_slack=res.mass_slack)
    assert p.exact >= len(seqs) - 3, p
    plen = gpu[0].cpu().numpy()
    assert plen.mean() > 0.5  # the draft tracks the target's logits


def test_bounded_wait_gives_up_and_the_next_call_is_clean():
    # the test-only flag withholds one shared-memory stage of the LM-head
    # kernel: the tensor-core issuer's bounded wait gives up (about a
    # second), the call completes with SPEC_STATUS_TIMEOUT, and the context
    # stays usable: the next call reports nothing and matches a clean call
    from speculative_decoding_verification_tree_gb300 import _lib
    w = synth.workload("lmhead_tree", B=2, V=2048, H=128, seed=17)
    hidden, wv, draft, q_row, toks, par = synth.lmhead_tree_inputs(w, "cuda")
    ws = api().workspace(_lib.SPEC_OP_TREE_LMHEAD, w.B, toks.shape[1], w.V)
    kw = dict(temperature=w.temperature, draft_kind=w.draft_kind,
              seed=w.decision_seed, ws=ws)
    clean = [x.clone() for x in api().spec_verify_tree_lmhead(
        hidden, wv, draft, q_row, toks, par, **kw)]
    assert api().spec_get_status(ws) == 0
    api().spec_verify_tree_lmhead(hidden, wv, draft, q_row, toks, par,
                                  flags=_lib.SPEC_FLAG_TEST_STALL, **kw)
    torch.cuda.synchronize()
    assert api().spec_get_status(ws) & _lib.SPEC_STATUS_TIMEOUT
    again = api().spec_verify_tree_lmhead(hidden, wv, draft, q_row, toks,
                                          par, **kw)
    torch.cuda.synchronize()
    assert api().spec_get_status(ws) == 0
    for a, b in zip(clean, again):
        assert torch.equal(a, b)
