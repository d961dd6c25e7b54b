"""The verification entry points inside a CUDA graph.

A serving loop captures its decode step once and replays it; every call of
the library only enqueues work on the caller's stream (launches, memsets)
and allocates nothing, so it can be captured.  Each case captures one call
into a torch CUDA graph with static inputs, outputs and workspace, writes
new inputs into the static tensors, replays, and checks that the replay's
outputs equal an eager call on the same inputs element by element (the
kernels are deterministic: no floating-point atomics, fixed reduction
orders) and the oracle's decisions."""

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


def _capture(fn):
    """Capture fn() (after two warm-up calls on a side stream); returns the
    graph and the outputs it writes."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.cpu(), y.cpu())


@pytest.mark.parametrize("name,B,K,V,top_k,top_p", [
    ("chain_sample", 1, 4, 32000, 0, 1.0),     # one launch, status word kept
    ("chain_sample", 24, 5, 32000, 0, 1.0),    # streaming kernels
    ("chain_topk", 8, 5, 32000, 50, 0.9),      # candidate lists
    ("greedy", 16, 8, 32000, 0, 1.0),          # argmax
])
def test_chain_call_replays_in_a_graph(name, B, K, V, top_k, top_p):
    from speculative_decoding_verification_tree_gb300 import _lib
    a = api()
    w = synth.workload(name, B=B, K=K, V=V, top_k=top_k, top_p=top_p,
                       seed=3)
    target, draft, toks = synth.chain_inputs(w, "cuda")
    ws = a.workspace(_lib.SPEC_OP_CHAIN, B, K, V)
    kw = dict(temperature=w.temperature, top_k=w.top_k, top_p=w.top_p,
              draft_kind=w.draft_kind, seed=w.decision_seed)
    g, out = _capture(lambda: a.spec_verify_chain(target, draft, toks, ws=ws,
                                                  **kw))
    # new inputs into the static tensors, then the replay
    w2 = synth.workload(name, B=B, K=K, V=V, top_k=top_k, top_p=top_p,
                        seed=4)
    t2, d2, k2 = synth.chain_inputs(w2, "cuda")
    target.copy_(t2)
    if draft is not None:
        draft.copy_(d2)
    toks.copy_(k2)
    g.replay()
    torch.cuda.synchronize()
    status = a.spec_get_status(ws)
    eager = a.spec_verify_chain(t2, d2, k2,
                                ws=a.workspace(_lib.SPEC_OP_CHAIN, B, K, V),
                                **kw)
    torch.cuda.synchronize()
    _same(out, eager)
    ref = verify_chain(np64(t2), None if d2 is None else np64(d2),
                       k2.cpu().numpy(), temperature=w.temperature,
                       top_k=w.top_k, top_p=w.top_p,
                       draft_kind=w.draft_kind, seed=w.decision_seed)
    if w.temperature > 0:
        compare_chain(out, ref, max_excluded=1)
        assert status == ref.status
    else:
        assert out[0].cpu().tolist() == ref.accepted.tolist()
        assert out[1].cpu().numpy().tolist() == ref.tokens.tolist()


def test_tree_call_replays_in_a_graph():
    from speculative_decoding_verification_tree_gb300 import _lib
    a = api()
    w = synth.workload("tree_static", B=4, V=32000)
    target, draft, q_row, toks, par = synth.tree_inputs(w, "cuda")
    N = toks.shape[1]
    ws = a.workspace(_lib.SPEC_OP_TREE, w.B, N, w.V)
    kw = dict(temperature=w.temperature, draft_kind=w.draft_kind,
              seed=w.decision_seed)
    g, out = _capture(lambda: a.spec_verify_tree(target, draft, q_row, toks,
                                                 par, ws=ws, **kw))
    w2 = synth.workload("tree_static", B=4, V=32000, seed=w.seed + 1)
    t2, d2, q2, k2, p2 = synth.tree_inputs(w2, "cuda")
    for dst, src in ((target, t2), (draft, d2), (q_row, q2), (toks, k2),
                     (par, p2)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    eager = a.spec_verify_tree(t2, d2, q2, k2, p2,
                               ws=a.workspace(_lib.SPEC_OP_TREE, w.B, N, w.V),
                               **kw)
    torch.cuda.synchronize()
    _same(out, eager)
    ref = verify_tree(np64(t2), np64(d2), q2.cpu().numpy(), k2.cpu().numpy(),
                      p2.cpu().numpy(), temperature=w.temperature,
                      draft_kind=w.draft_kind, seed=w.decision_seed)
    compare_tree(out, ref, max_excluded=1)
