"""Seeded synthetic inputs shaped like the workloads the pages describe.

Shared by the CUDA path's tests / bench and by the oracle's tests.  This module
holds none of the verification arithmetic: it draws logits, and it stands in
for the draft model (drawing draft tokens from the draft distribution with
torch's own softmax / topk / multinomial primitives), which is outside the
verification path.  Everything is a pure function of its seed.

Workloads (sizes and distributions):
  chain_sample  B=1,  K=4, V=32000 fp32; target ~ N(0, 2^2); draft = target +
                N(0, 0.7^2); T = 1; draft tokens ~ q (generator seed 0);
                decisions use Philox seed 1.
  chain_topk    B=64, K=5, V=32000 bf16; target ~ N(0, 3^2); draft = target +
                N(0, 1); T = 0.7, top-k 50, top-p 0.9; tokens ~ transformed q.
  greedy        B=256, K=8, V=128256 bf16 ~ N(0, 2.5^2); draft tokens =
                argmax(target + N(0, 1.5^2)).
  tree_static   B=32, 60-node static tree, depth 6, branching (4,3,2,2,1,1)
                filled to level widths (4,12,16,14,8,6); target bf16 [B,61,V]
                ~ N(0, 2^2); draft probs fp32 = softmax(target + N(0, 0.8^2));
                T = 1; sibling tokens drawn without replacement from q.
  lmhead_tree   the tree_static tree, batch and draft rule, with the target
                logits coming from hidden states: hidden [B,61,H=4096] bf16
                ~ N(0, 1), LM head W [V,H] bf16 ~ N(0, (2/sqrt(H))^2) (logits
                of std about 2); the stand-in drafter perturbs the float32
                product h W^T (torch matmul, input generation only).
  eagle2        B=128, V=128256 bf16; draft rows [B,51,V] ~ N(0, 2.5^2);
                target row = its draft row + N(0, 1) (rows without a draft
                row: fresh N(0, 2.5^2) + N(0, 1)); depth 6, 10 children, keep
                10 per layer, total 60; T = 0.8.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

V_LLAMA3 = 128256


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int            # chain: drafts per sequence; tree: drafted nodes N
    V: int
    target_dtype: torch.dtype
    draft_dtype: torch.dtype
    temperature: float
    top_k: int = 0
    top_p: float = 1.0
    draft_kind: str = "logits"
    target_std: float = 2.0
    draft_noise: float = 0.7
    seed: int = 1234           # logits generator seed
    draft_seed: int = 0        # drafter's sampling seed
    decision_seed: int = 1     # Philox key of the verifier's uniforms
    branching: tuple = field(default=())
    widths: tuple = field(default=())
    depth: int = 6
    topk: int = 10
    width: int = 10
    total: int = 60
    H: int = 0                 # hidden size (LM-head workloads)


WORKLOADS = {
    "chain_sample": Workload("chain_sample", 1, 4, 32000, torch.float32,
                             torch.float32, 1.0, target_std=2.0,
                             draft_noise=0.7, seed=1234),
    "chain_topk": Workload("chain_topk", 64, 5, 32000, torch.bfloat16,
                           torch.bfloat16, 0.7, top_k=50, top_p=0.9,
                           target_std=3.0, draft_noise=1.0, seed=1235),
    "greedy": Workload("greedy", 256, 8, V_LLAMA3, torch.bfloat16,
                       torch.bfloat16, 0.0, target_std=2.5, draft_noise=1.5,
                       seed=1236),
    "tree_static": Workload("tree_static", 32, 60, V_LLAMA3, torch.bfloat16,
                            torch.float32, 1.0, draft_kind="probs",
                            target_std=2.0, draft_noise=0.8, seed=1237,
                            branching=(4, 3, 2, 2, 1, 1),
                            widths=(4, 12, 16, 14, 8, 6)),
    "lmhead_tree": Workload("lmhead_tree", 32, 60, V_LLAMA3, torch.bfloat16,
                            torch.float32, 1.0, draft_kind="probs",
                            target_std=2.0, draft_noise=0.8, seed=1239,
                            branching=(4, 3, 2, 2, 1, 1),
                            widths=(4, 12, 16, 14, 8, 6), H=4096),
    "eagle2": Workload("eagle2", 128, 60, V_LLAMA3, torch.bfloat16,
                       torch.bfloat16, 0.8, target_std=2.5, draft_noise=1.0,
                       seed=1238),
}


def workload(name: str, **overrides) -> Workload:
    return replace(WORKLOADS[name], **overrides)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device,
                       dtype=torch.float32) * std


# ----------------------------------------------------------------- drafter
def _sample(q, m, g, replacement):
    """Draw m tokens per row from q.  The probabilities are checked on the
    host first, so a bad distribution raises here instead of tripping a
    device-side assert inside torch's sampler."""
    ok = torch.isfinite(q).all() & (q >= 0).all() & (q.sum(-1) > 0).all()
    if not bool(ok):
        raise ValueError("draft distribution is not a valid probability row")
    if not replacement and int((q > 0).sum(-1).min()) < m:
        replacement = True  # too few tokens for distinct siblings
    return torch.multinomial(q, m, replacement=replacement, generator=g)


def _draft_dist(logits, w: Workload):
    """Draft model's sampling distribution (stand-in drafter; torch ops).
    Temperature must be positive (greedy drafting uses top-m instead)."""
    if not w.temperature > 0:
        raise ValueError("sampling drafter needs temperature > 0")
    z = logits.float()
    if w.draft_kind == "probs":
        z = torch.log(z)
    z = z / w.temperature
    if w.top_k > 0 and w.top_k < z.shape[-1]:
        # exactly k tokens; ties at the k-th value go to the lower index
        order = torch.sort(z, dim=-1, descending=True, stable=True).indices
        keep = torch.zeros_like(z, dtype=torch.bool).scatter_(
            -1, order[..., :w.top_k], True)
        z = torch.where(keep, z, torch.full_like(z, float("-inf")))
    probs = torch.softmax(z, dim=-1)
    if w.top_p < 1.0:
        sp, idx = torch.sort(probs, dim=-1, descending=True, stable=True)
        cum = torch.cumsum(sp, dim=-1)
        drop = (cum - sp) >= w.top_p
        sp = torch.where(drop, torch.zeros_like(sp), sp)
        probs = torch.zeros_like(probs).scatter_(-1, idx, sp)
        probs = probs / probs.sum(-1, keepdim=True)
    return probs


# ------------------------------------------------------------------ chains
def chain_inputs(w: Workload, device="cpu"):
    """target [B,K+1,V], draft [B,K,V] (None for greedy), tokens [B,K]."""
    g = _gen(device, w.seed)
    B, K, V = w.B, w.K, w.V
    tgt = _normal((B, K + 1, V), w.target_std, g, device)
    noisy = tgt[:, :K] + _normal((B, K, V), w.draft_noise, g, device)
    gd = _gen(device, w.draft_seed)
    if w.temperature == 0:
        tokens = torch.argmax(noisy, dim=-1).to(torch.int32)
        return tgt.to(w.target_dtype), None, tokens.contiguous()
    target = tgt.to(w.target_dtype)
    if w.draft_kind == "probs":
        draft = torch.softmax(noisy, dim=-1).to(w.draft_dtype)
    else:
        draft = noisy.to(w.draft_dtype)
    q = _draft_dist(draft, w).reshape(B * K, V)
    tokens = _sample(q, 1, gd, False).reshape(B, K)
    return target, draft, tokens.to(torch.int32).contiguous()


# ------------------------------------------------------------- static tree
def static_tree(w: Workload, device="cpu"):
    """Parent array of the static tree (shared by the batch), BFS order.
    Level d offers branching[d-1] child slots under each node of level d-1;
    widths[d-1] of them are filled, chosen without replacement by a seeded
    generator (seed 2) and kept in slot order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(2)
    parent = []
    prev = [-1]  # node indices of the previous level (-1 = root)
    for br, wd in zip(w.branching, w.widths):
        slots = [(p, c) for p in prev for c in range(br)]
        assert wd <= len(slots)
        pick = torch.randperm(len(slots), generator=g)[:wd].sort().values
        level = []
        for i in pick.tolist():
            p, _ = slots[i]
            level.append(len(parent))
            parent.append(p)
        prev = level
    return torch.tensor(parent, dtype=torch.int32, device=device)


def tree_inputs(w: Workload, device="cpu", parent=None):
    """target [B,N+1,V], draft [B,N+1,V] (every row has a draft row),
    q_row [B,N+1], node_tokens [B,N], parent [B,N]."""
    if parent is None:
        parent = static_tree(w, device)
    parent = parent.to(device)
    N = parent.numel()
    B, V = w.B, w.V
    g = _gen(device, w.seed)
    tgt = _normal((B, N + 1, V), w.target_std, g, device)
    noisy = tgt + _normal((B, N + 1, V), w.draft_noise, g, device)
    target = tgt.to(w.target_dtype)
    del tgt
    draft, q_row, tokens, par = _tree_draft(w, noisy, parent, device)
    return target, draft, q_row, tokens, par


def lmhead_tree_inputs(w: Workload, device="cpu", parent=None):
    """hidden [B,N+1,H] bf16, w_vocab [V,H] bf16, draft [B,N+1,V], q_row,
    node_tokens [B,N], parent [B,N] (the static tree)."""
    if parent is None:
        parent = static_tree(w, device)
    parent = parent.to(device)
    N = parent.numel()
    B, V, H = w.B, w.V, w.H
    g = _gen(device, w.seed)
    hidden = _normal((B, N + 1, H), 1.0, g, device).to(torch.bfloat16)
    wv = _normal((V, H), w.target_std / H ** 0.5, g, device).to(
        torch.bfloat16)
    # the stand-in drafter sees a perturbed copy of the target's logits
    noisy = torch.matmul(hidden.float(), wv.float().t())
    noisy += _normal((B, N + 1, V), w.draft_noise, g, device)
    draft, q_row, tokens, par = _tree_draft(w, noisy, parent, device)
    return hidden, wv, draft, q_row, tokens, par


def _tree_draft(w: Workload, noisy, parent, device):
    """Draft rows from the drafter's logits, the identity q_row, sibling
    tokens drawn without replacement from q, and the batch's parent rows."""
    B, N1, V = noisy.shape
    N = N1 - 1
    if w.draft_kind == "probs":
        draft = torch.softmax(noisy, dim=-1).to(w.draft_dtype)
    else:
        draft = noisy.to(w.draft_dtype)
    del noisy
    q_row = torch.arange(N + 1, dtype=torch.int32, device=device)
    q_row = q_row.unsqueeze(0).expand(B, N + 1).contiguous()
    # siblings drawn without replacement from the parent row's q
    gd = _gen(device, w.draft_seed)
    tokens = torch.empty(B, N, dtype=torch.int32, device=device)
    pl = parent.tolist()
    kids = {}
    for j, p in enumerate(pl):
        kids.setdefault(p + 1, []).append(j)
    for r, ks in kids.items():
        if w.temperature > 0:
            q = _draft_dist(draft[:, r], w)
            draws = _sample(q, len(ks), gd, False)
        else:  # greedy drafter: the len(ks) most likely tokens
            draws = torch.topk(draft[:, r].float(), len(ks), dim=-1).indices
        tokens[:, ks] = draws.to(torch.int32)
    par = parent.unsqueeze(0).expand(B, N).contiguous()
    return draft, q_row, tokens, par


# ------------------------------------------------------------------ EAGLE-2
def eagle2_draft(w: Workload, device="cpu"):
    R = 1 + (w.depth - 1) * w.width
    g = _gen(device, w.seed)
    return _normal((w.B, R, w.V), w.target_std, g, device).to(w.draft_dtype)


def eagle2_target(w: Workload, draft, q_row, device="cpu"):
    """Target rows for the reranked tree: draft row + N(0, 1) where the tree
    row has a draft row, fresh N(0, std^2) + N(0, 1) elsewhere."""
    B, M1 = q_row.shape
    if int(q_row.max()) >= draft.shape[1] or int(q_row.min()) < -1:
        raise ValueError("q_row names a draft row that does not exist")
    g = _gen(device, w.seed + 1)
    fresh = _normal((B, M1, w.V), w.target_std, g, device)
    noise = _normal((B, M1, w.V), w.draft_noise, g, device)
    idx = q_row.clamp(min=0).long()
    base = torch.gather(draft.float(), 1,
                        idx.unsqueeze(-1).expand(B, M1, w.V))
    base = torch.where((q_row >= 0).unsqueeze(-1), base, fresh)
    return (base + noise).to(w.target_dtype)
