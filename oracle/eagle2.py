"""EAGLE-2 dynamic draft tree: expand and rerank (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

From "EAGLE-2: Faster Inference of Language Models with Dynamic Draft Trees"
(papercache notes):

* §4.1 value: a node's global acceptance estimate is the product over its
  root path of the draft confidences c_j (the equation itself is lost on the
  page; the text around it defines it).  We carry it as the sum of log q,
  which orders nodes identically without underflow.
* §4.1 expand: at each layer the top-k nodes of the newest layer by value are
  fed to the draft model, and each one's draft distribution adds its most
  probable tokens as children.
* §4.2 rerank: all drafted nodes are reranked by value and the top-m kept;
  ties prefer the shallower node, so the kept set stays a connected tree;
  the kept nodes are flattened (parents before children) and given the
  ancestor-only attention mask.

Synthetic harness (the draft forward between layers is outside this path):
``draft`` holds every draft row up front, row 0 for the root and row
1 + (d-1)*W + r for the r-th kept node of layer d (d = 1 .. L-1).

Readings taken where the pages are silent: confidence = q after the temperature
transform; children of a row are its ``topk`` most probable tokens (ties to the
lower index); layer keep and rerank order by (value desc, depth asc, candidate
id asc) with candidate id = (layer, parent rank, child rank).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .sampling import transform_logits
from .tree import tree_mask


@dataclass
class Eagle2Result:
    node_tokens: np.ndarray   # [B, M] int32
    parent: np.ndarray        # [B, M] int32, -1 = child of the root
    q_row: np.ndarray         # [B, M+1] int32, draft row per tree row or -1
    value: np.ndarray         # [B, M] float64, sum of log q along the path
    mask: np.ndarray          # [B, M, M] uint8
    candidates: list          # per b: list of candidate dicts (for tests)


def _row_children(row, temperature, topk):
    q, _ = transform_logits(row, temperature)
    order = np.lexsort((np.arange(q.size), -q))[:topk]
    with np.errstate(divide="ignore"):
        return [(int(x), float(np.log(q[x])) if q[x] > 0 else -np.inf)
                for x in order]


def expand_rerank(draft, *, temperature: float, depth: int = 6,
                  topk: int = 10, width: int = 10,
                  total: int = 60) -> Eagle2Result:
    draft = np.asarray(draft)
    B, R, V = draft.shape
    L, W, M = depth, width, total
    assert R >= 1 + (L - 1) * W
    toks = np.full((B, M), -1, dtype=np.int32)
    par = np.full((B, M), -1, dtype=np.int32)
    qrow = np.full((B, M + 1), -1, dtype=np.int32)
    val = np.full((B, M), np.nan, dtype=np.float64)
    all_cands = []
    for b in range(B):
        cands = []  # dicts: token, value, depth, id, parent (cand index)
        # layer 1: children of the root, draft row 0
        layer = []
        for c, (x, lq) in enumerate(_row_children(draft[b, 0], temperature,
                                                  topk)):
            layer.append(dict(token=x, value=lq, depth=1, id=(1, 0, c),
                              parent=None, row=None))
        for d in range(1, L + 1):
            cands.extend(layer)
            kept = sorted(layer, key=lambda n: (-n["value"], n["depth"],
                                                n["id"]))[:W]
            if d == L:
                break
            nxt = []
            for r, node in enumerate(kept):
                node["row"] = 1 + (d - 1) * W + r
                for c, (x, lq) in enumerate(_row_children(
                        draft[b, node["row"]], temperature, topk)):
                    nxt.append(dict(token=x, value=node["value"] + lq,
                                    depth=d + 1, id=(d + 1, r, c),
                                    parent=node, row=None))
            layer = nxt
        assert M <= len(cands)
        sel = sorted(cands, key=lambda n: (-n["value"], n["depth"],
                                           n["id"]))[:M]
        pos = {id(n): i for i, n in enumerate(sel)}
        qrow[b, 0] = 0
        for i, n in enumerate(sel):
            toks[b, i] = n["token"]
            val[b, i] = n["value"]
            par[b, i] = -1 if n["parent"] is None else pos[id(n["parent"])]
            qrow[b, i + 1] = -1 if n["row"] is None else n["row"]
        all_cands.append(cands)
    mask, _ = tree_mask(par)
    return Eagle2Result(toks, par, qrow, val, mask, all_cands)
