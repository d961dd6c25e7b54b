"""Acceptance records on the GPU vs the oracle (integer records bit-exact,
confidence sums to rel 1e-12)."""

import numpy as np
import pytest
import torch

import synth
from oracle import stats as ostats
from tests._parity import lib_ready

pytestmark = pytest.mark.gpu

INT_FIELDS = ("len_hist", "node_tested", "node_accepted", "depth_tested",
              "depth_accepted", "calib_tested", "calib_accepted")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _random_parent(rng, n):
    return np.array([-1 if j == 0 or rng.random() < 0.15
                     else int(rng.integers(max(0, j - 8), j))
                     for j in range(n)], dtype=np.int32)


def _rounds(rng, par, B, invalid=0.1):
    """Per round: path to a random node (or empty), some made invalid."""
    n = par.shape[1]
    count = np.zeros(B, dtype=np.int32)
    nodes = np.full((B, n), -1, dtype=np.int32)
    for b in range(B):
        if rng.random() < 0.15:
            continue
        j, chain = int(rng.integers(0, n)), []
        while j >= 0:
            chain.append(j)
            j = int(par[b, j])
        chain.reverse()
        count[b] = len(chain)
        nodes[b, :len(chain)] = chain
        if rng.random() < invalid:
            kind = int(rng.integers(0, 4))
            if kind == 0:
                count[b] = n + 1
            elif kind == 1:
                nodes[b, 0] = n  # out of range
            elif kind == 2 and len(chain) >= 2:
                nodes[b, 1] = nodes[b, 0]  # not a child of its predecessor
            else:
                count[b] = -3
    return count, nodes


def _confidence(rng, B, n):
    c = rng.random((B, n)).astype(np.float32)
    special = np.array([np.nan, -0.25, 1.0, 1.5, 0.0, 0.05, 0.5, 0.95],
                       dtype=np.float32)
    pick = rng.random((B, n)) < 0.1
    c[pick] = special[rng.integers(0, special.size, size=int(pick.sum()))]
    return c


def _gpu(count, parent, nodes, conf, n, nbins, out=None):
    d = lambda a: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a)).cuda()
    r = api().spec_accept_stats(d(count), d(parent), d(nodes), d(conf), n=n,
                                nbins=nbins, out=out)
    torch.cuda.synchronize()
    return r


def _check(rec, st, fields=INT_FIELDS):
    for f in fields:
        assert np.array_equal(rec[f].cpu().numpy(), getattr(st, f)), f
    assert int(rec["invalid"].item()) == st.invalid
    cs = rec["calib_conf_sum"].cpu().numpy()
    assert np.allclose(cs, st.calib_conf_sum, rtol=1e-12, atol=0)


# n <= 64: one warp per round (B = 6000 makes warps take several rounds);
# above: one CTA per round (B = 400 makes CTAs take several rounds)
@pytest.mark.parametrize("n,B,nbins", [(1, 5, 4), (7, 40, 20), (33, 50, 7),
                                       (60, 32, 20), (60, 700, 50),
                                       (60, 6000, 20), (64, 100, 20),
                                       (65, 30, 20), (100, 400, 10),
                                       (200, 64, 10), (300, 50, 1024),
                                       (1024, 9, 20), (1024, 5, 1024)])
def test_tree_records(n, B, nbins):
    rng = np.random.default_rng(n * 1000 + B)
    par = np.stack([_random_parent(rng, n) for _ in range(B)])
    count, nodes = _rounds(rng, par, B)
    conf = _confidence(rng, B, n)
    rec = _gpu(count, par, nodes, conf, n, nbins)
    st = ostats.accept_stats(count, par, nodes, conf, n, nbins)
    _check(rec, st)


def test_forward_parent_arrays_are_invalid_rounds():
    rng = np.random.default_rng(4)
    n, B = 12, 20
    par = np.stack([_random_parent(rng, n) for _ in range(B)])
    count, nodes = _rounds(rng, par, B, invalid=0.0)
    par[3, 5] = 7       # points forward
    par[8, 0] = 0       # points to itself
    par[11, 4] = -2     # below -1
    rec = _gpu(count, par, nodes, None, n, 4)
    st = ostats.accept_stats(count, par, nodes, None, n, 4)
    assert st.invalid >= 3
    _check(rec, st)


@pytest.mark.parametrize("n,B", [(4, 9), (8, 256), (40, 6000), (64, 50),
                                 (100, 400)])
def test_chain_records(n, B):
    rng = np.random.default_rng(n + B)
    count = rng.integers(-2, n + 3, size=B).astype(np.int32)
    conf = _confidence(rng, B, n)
    rec = _gpu(count, None, None, conf, n, 20)
    st = ostats.accept_stats(count, None, None, conf, n, 20)
    _check(rec, st)


def test_records_accumulate_and_skip_missing_entries():
    rng = np.random.default_rng(12)
    n, B, nb = 30, 100, 16
    par = np.stack([_random_parent(rng, n)] * B)
    out = api().accept_stats_records(n, nb)
    out["depth_tested"] = None
    out["calib_conf_sum"] = None
    st = ostats.empty(n, nb)
    for call in range(2):
        count, nodes = _rounds(rng, par, B)
        conf = _confidence(rng, B, n)
        _gpu(count, par, nodes, conf, n, nb, out=out)
        ostats.accept_stats(count, par, nodes, conf, n, nb, into=st)
    fields = [f for f in INT_FIELDS if f != "depth_tested"]
    for f in fields:
        assert np.array_equal(out[f].cpu().numpy(), getattr(st, f)), f
    assert int(out["invalid"].item()) == st.invalid


def test_records_of_verified_static_trees_full_size():
    # the 60-node static tree at B = 32, V = 128256: records computed from
    # spec_verify_tree's own outcomes, confidence = q of each drafted token
    w = synth.workload("tree_static")
    target, draft, q_row, toks, par = synth.tree_inputs(w, "cuda")
    plen, pnodes, _, _ = api().spec_verify_tree(
        target, draft, q_row, toks, par, temperature=w.temperature,
        draft_kind=w.draft_kind, seed=w.decision_seed)
    rows = (par.long() + 1).unsqueeze(-1)                   # parent's row
    q = torch.gather(draft, 1, rows.expand(-1, -1, draft.shape[-1]))
    conf = torch.gather(q, 2, toks.long().unsqueeze(-1)).squeeze(-1)
    conf = (conf / q.sum(-1)).float().contiguous()
    del q
    N = toks.shape[1]
    rec = api().spec_accept_stats(plen, par, pnodes, conf, n=N, nbins=20)
    torch.cuda.synchronize()
    st = ostats.accept_stats(plen.cpu().numpy(), par.cpu().numpy(),
                             pnodes.cpu().numpy(), conf.cpu().numpy(), N, 20)
    _check(rec, st)
    assert st.invalid == 0 and st.len_hist.sum() == w.B
    assert st.node_tested[:4].sum() >= w.B  # the root's first child always


def test_records_of_verified_chains():
    w = synth.workload("chain_topk")
    target, draft, toks = synth.chain_inputs(w, "cuda")
    acc, _, _ = api().spec_verify_chain(
        target, draft, toks, temperature=w.temperature, top_k=w.top_k,
        top_p=w.top_p, seed=w.decision_seed)
    q = synth._draft_dist(draft, w)
    conf = torch.gather(q, 2, toks.long().unsqueeze(-1)).squeeze(-1)
    conf = conf.float().contiguous()
    rec = api().spec_accept_stats(acc, n=w.K, nbins=10, confidence=conf)
    torch.cuda.synchronize()
    st = ostats.accept_stats(acc.cpu().numpy(), None, None,
                             conf.cpu().numpy(), w.K, 10)
    _check(rec, st)
    assert st.node_tested[0] == w.B
