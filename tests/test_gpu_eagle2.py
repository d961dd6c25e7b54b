"""EAGLE-2 expand + rerank (and the full dynamic-tree pipeline) vs the oracle.

Node values are float32 sums of log q on the GPU and float64 in the oracle, so
the selection can legitimately differ where two candidate values lie within
1e-5 of each other at a layer-keep or rerank boundary.  Where the oracle sees
no such near tie the GPU tree must match exactly (tokens, parents, q_row);
otherwise it must be a valid EAGLE-2 tree for the oracle's values.
"""

import numpy as np
import pytest
import torch

import synth
from oracle.eagle2 import expand_rerank
from oracle.sampling import transform_logits
from oracle.tree import tree_mask, verify_tree
from tests._parity import compare_tree, lib_ready, np64

pytestmark = pytest.mark.gpu
VAL_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _near_ties(cands, W, M, L):
    """Does any keep / rerank boundary (or the order of kept nodes) involve
    values closer than VAL_TOL?"""
    def close(x, y):
        a, b = x["value"], y["value"]
        if a == b and (x["parent"] is y["parent"] or x["parent"] is y
                       or y["parent"] is x):
            # siblings with equal logits, or a child of confidence 1: the
            # float32 values are equal too, so the tie rule decides exactly
            return False
        return abs(a - b) <= VAL_TOL * max(1.0, abs(a), abs(b))
    for d in range(1, L):
        layer = sorted([c for c in cands if c["depth"] == d],
                       key=lambda c: (-c["value"], c["id"]))
        for i in range(min(W, len(layer) - 1)):
            if close(layer[i], layer[i + 1]):
                return True
    allc = sorted(cands, key=lambda c: (-c["value"], c["depth"], c["id"]))
    for i in range(min(M, len(allc) - 1)):
        if close(allc[i], allc[i + 1]):
            return True
    return False


def _check_valid(draft, b, T, topk, tok, par, qrow, val):
    """The GPU tree is a connected EAGLE-2 tree whose values are the oracle's
    log-probability sums (float64 recomputation)."""
    M = tok.shape[0]
    lq = {}
    for j in range(M):
        p = par[j]
        assert -1 <= p < j
        row = 0 if p < 0 else qrow[p + 1]
        assert row >= 0, "a node's parent must have been expanded"
        if row not in lq:
            q, _ = transform_logits(draft[b, row], T)
            lq[row] = (np.log(np.where(q > 0, q, 1e-300)), q)
        logq, q = lq[row]
        top = np.lexsort((np.arange(q.size), -q))[:topk]
        assert tok[j] in top
        want = (0.0 if p < 0 else val[p]) + logq[tok[j]]
        assert abs(val[j] - want) <= 1e-4 * max(1.0, abs(want))


def _run(w, draft):
    L, K, W, M = w.depth, w.topk, w.width, w.total
    tok, par, qrow, val, mask = api().spec_eagle2_expand_rerank(
        draft, temperature=w.temperature, depth=L, topk=K, width=W, total=M)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in (tok, par, qrow, val, mask)]


def _compare(w, draft, gpu, seqs):
    tok, par, qrow, val, mask = gpu
    d64 = np64(draft[seqs])
    ref = expand_rerank(d64, temperature=w.temperature, depth=w.depth,
                        topk=w.topk, width=w.width, total=w.total)
    near = 0
    for i, b in enumerate(seqs):
        want_mask, _ = tree_mask(par[b:b + 1])
        assert np.array_equal(mask[b], want_mask[0])
        if _near_ties(ref.candidates[i], w.width, w.total, w.depth):
            near += 1
            _check_valid(d64, i, w.temperature, w.topk, tok[b], par[b],
                         qrow[b], val[b])
            continue
        assert np.array_equal(tok[b], ref.node_tokens[i]), b
        assert np.array_equal(par[b], ref.parent[i]), b
        assert np.array_equal(qrow[b], ref.q_row[i]), b
        np.testing.assert_allclose(val[b], ref.value[i], rtol=1e-5, atol=1e-5)
    return near


@pytest.mark.parametrize("V,dt", [(64, torch.float32), (1000, torch.bfloat16),
                                  (4099, torch.float32),
                                  (32000, torch.bfloat16)])
def test_expand_rerank_small_vocab(V, dt):
    w = synth.workload("eagle2", B=6, V=V, draft_dtype=dt, seed=V)
    draft = synth.eagle2_draft(w, "cuda")
    gpu = _run(w, draft)
    near = _compare(w, draft, gpu, list(range(w.B)))
    assert near <= 2


def test_expand_rerank_other_shapes():
    w = synth.workload("eagle2", B=5, V=3000, depth=3, topk=4, width=3,
                       total=12, seed=4)
    draft = synth.eagle2_draft(w, "cuda")
    _compare(w, draft, _run(w, draft), list(range(5)))
    w = synth.workload("eagle2", B=3, V=500, depth=1, topk=7, width=2,
                       total=5, seed=5)
    draft = synth.eagle2_draft(w, "cuda")
    _compare(w, draft, _run(w, draft), list(range(3)))


def test_expand_rerank_ties_and_certain_tokens():
    # integer logits: many exact ties (broken by token index, then depth,
    # then candidate id) and rows whose top token has probability 1
    w = synth.workload("eagle2", B=3, V=300, depth=4, topk=3, width=3,
                       total=20, seed=6)
    R = 1 + (w.depth - 1) * w.width
    g = torch.Generator(device="cpu").manual_seed(0)
    d = torch.randint(-3, 3, (w.B, R, w.V), generator=g).float()
    d[1, 2] = float("-inf")
    d[1, 2, 17] = 0.0
    draft = d.to(torch.bfloat16).cuda()
    _compare(w, draft, _run(w, draft), list(range(w.B)))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_expand_rerank_ties_aligned_rows(dt):
    # aligned rows (V % 8 == 0, the bound-and-rescan path): logits on a 1/4
    # grid give exact ties among the top few (ranked by index); rows of small
    # integers tie thousands of logits at the top (more candidates than the
    # rescan keeps: the general top-k takes the row)
    w = synth.workload("eagle2", B=3, V=32000, depth=3, topk=10, width=4,
                       total=20, seed=7, draft_dtype=dt)
    R = 1 + (w.depth - 1) * w.width
    g = torch.Generator(device="cpu").manual_seed(1)
    d = torch.round(torch.randn(w.B, R, w.V, generator=g) * 2.5 * 4) / 4
    d[2] = torch.randint(-3, 3, (R, w.V), generator=g).float()
    draft = d.to(dt).cuda()
    _compare(w, draft, _run(w, draft), list(range(w.B)))


def test_eagle2_full_pipeline_sampled():
    # B=128, V=128256 bf16: expand + rerank + mask, then tree verification at
    # T = 0.8 with target = draft row + noise, compared on sampled sequences
    w = synth.workload("eagle2")
    draft = synth.eagle2_draft(w, "cuda")
    tok, par, qrow, val, mask = api().spec_eagle2_expand_rerank(
        draft, temperature=w.temperature)
    seqs = list(range(0, w.B, 8))  # 16 of the 128 sequences
    gpu = [x.cpu().numpy() for x in (tok, par, qrow, val, mask)]
    _compare(w, draft, gpu, seqs)
    target = synth.eagle2_target(w, draft, qrow, "cuda")
    out = api().spec_verify_tree(target, draft, qrow, tok, par,
                                 temperature=w.temperature,
                                 seed=w.decision_seed)
    torch.cuda.synchronize()
    ref = verify_tree(np64(target[seqs]), np64(draft[seqs]),
                      qrow[seqs].cpu().numpy(), tok[seqs].cpu().numpy(),
                      par[seqs].cpu().numpy(), temperature=w.temperature,
                      seed=w.decision_seed, batch_ids=seqs)
    p = compare_tree(out, ref, seqs=seqs, max_excluded=2)
    assert p.exact >= len(seqs) - 3, p
    plen = out[0].cpu().numpy()
    assert plen.mean() > 0.5  # the synthetic target tracks the draft


@pytest.mark.parametrize("V,dt,B", [(32000, torch.bfloat16, 12),
                                    (128256, torch.bfloat16, 128),
                                    (4099, torch.float32, 6)])
def test_eagle2_verify_with_expand_normalisers(V, dt, B):
    # the expand writes each draft row's log2 normaliser; tree verification
    # then leaves the draft rows out of its first pass (aligned rows) or
    # ignores them (the general kernel) and must still match the oracle
    w = synth.workload("eagle2", B=B, V=V, draft_dtype=dt, seed=V + 11)
    draft = synth.eagle2_draft(w, "cuda")
    R = draft.shape[1]
    lse = torch.full((B, R), float("nan"), dtype=torch.float32, device="cuda")
    tok, par, qrow, val, mask = api().spec_eagle2_expand_rerank(
        draft, temperature=w.temperature, draft_lse=lse)
    torch.cuda.synchronize()
    # q = 2^(z log2(e) / T - lse) is a distribution (float64 recomputation)
    kt = np.log2(np.e) / w.temperature
    L = lse.cpu().numpy().astype(np.float64)
    for b, r in [(0, 0), (B - 1, R - 1), (B // 2, R // 2)]:
        z = np64(draft[b, r])
        assert abs(np.exp2(z * kt - L[b, r]).sum() - 1.0) < 3e-5, (b, r)
    target = synth.eagle2_target(w, draft, qrow, "cuda")
    out = api().spec_verify_tree(target, draft, qrow, tok, par,
                                 temperature=w.temperature,
                                 seed=w.decision_seed, draft_lse=lse)
    torch.cuda.synchronize()
    seqs = list(range(B)) if B <= 12 else [1, 64, 126]
    ref = verify_tree(np64(target[seqs]), np64(draft[seqs]),
                      qrow[seqs].cpu().numpy(), tok[seqs].cpu().numpy(),
                      par[seqs].cpu().numpy(), temperature=w.temperature,
                      seed=w.decision_seed, batch_ids=seqs)
    compare_tree(out, ref, seqs=seqs)
