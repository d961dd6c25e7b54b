"""Plain CPU float64 oracle for speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously-correct
restatement of what the verification path computes, written from the method's
definition and nothing else.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA product path never imports, links or executes anything here, and
nothing here imports the product package: the two share no code.  The only
module both sides use is ``synth`` (seeded input generators, which hold none of
the verification arithmetic).

Sources (cited by page title and section throughout):

* "投机解码与 EAGLE" (aiknowledge.cn lesson): the four-step draft/verify loop,
  the exactness rule ("精确性规则"), the greedy simplification, expected tokens
  per target pass ("期望加速比"), tree drafts ("EAGLE:树形草稿").
* "064 · 投机解码：小模型先起草，大模型怎样并行验收而不改变分布" (Leviathan et al.
  analysis): a(x) and r(x) (section 二), acceptance mass = 1 - TV
  ("接受率等于两个分布重叠的质量"), the two-token worked examples, the verify
  listing (section 三), and that p, q include temperature / top-k / nucleus.
* "EAGLE-2: Faster Inference of Language Models with Dynamic Draft Trees"
  (papercache notes): the norm(max(0, p - p_hat)) rule (§2.1), tree drafts
  (§2.2), value = product of confidences (§4.1), expand (§4.1), rerank and the
  ancestor-only attention mask (§4.2).
* "Việc giải mã giả định và EAGLE-3" and "Descodación especulativa Draft,
  Verificar, Replicar" (aiengineeringfromscratch lessons; both swap the names
  p and q): the q = 0 accept rule ("Bước 1" / "Paso 1") and the zero-mass
  residual fallback ("Bước 2").

Convention everywhere: p = target (verifier) distribution, q = draft.

Parity status per function is listed in ``PINS`` below; every function is
pinned by tests in ``tests/test_oracle_*.py`` except where marked
"parity unpinned".
"""

PINS = {
    "philox.philox4x32_10": "equal to an independent library implementation "
    "(Triton's tl.philox, ten rounds, run as a black box in its CPU "
    "interpreter) on extreme and random keys and counters; structural "
    "(bijection per key) + uniformity chi-square",
    "sampling.transform": "brute force vs stable sort on V<=64; softmax closed "
    "forms",
    "sampling.residual / accept_prob": "worked examples of the Leviathan "
    "analysis page (exact Fractions); exact losslessness on V<=4",
    "chain.verify_chain": "Monte-Carlo losslessness (KL, chi-square); "
    "E[tokens] closed form; greedy reduces to numpy.argmax",
    "tree.tree_mask": "brute-force ancestor sets; chain -> lower triangular",
    "tree.verify_tree": "exact losslessness of the sibling recursion (2x3 and "
    "[2,2,2] trees, Fractions); Monte-Carlo first/second-token marginals; "
    "chain special case equals verify_chain",
    "eagle2.expand_rerank": "brute force over all candidates with sorted(); "
    "connectivity invariant",
    "analysis": "E[tokens], speedup and op-count values printed on the pages",
    "kv.kv_commit": "the rollback exercise of the Spanish page (prefix 10, "
    "5 drafts, rejection at the third); the logical-length rule of the "
    "Vietnamese page; in-place path-order copy equals the alias-free gather; "
    "the committed entries of a tree are the tokens verify_tree emits",
    "stats.accept_stats": "hand-worked tree and chain example "
    "(tests/golden/accept_stats_example.txt); tested set equal to a "
    "step-by-step simulation of the decisions over every outcome of small "
    "trees; truncated-geometric lengths and E[tokens] of an i.i.d. chain; a "
    "calibrated drafter on the diagonal; first- and second-sibling rates of "
    "verify_tree equal to their exact values",
    "attention.tree_attention": "torch scaled_dot_product_attention "
    "(float64) with the mask written out per position, grouped-query heads "
    "included; the chain case equals causal attention; a root child without "
    "prefix returns its own value; other branches and the prefix order do "
    "not change a node's output",
    "lmhead.lm_head_logits / bf16_round": "bf16 rounding equal to torch's "
    "float32 -> bfloat16 conversion (ties included); neighbours bracket the "
    "value one bf16 unit apart; exact logits equal rational dot products; "
    "the accumulation bound covers an explicit float32 summation in groups "
    "of 16",
    "lmhead.verify_tree_lmhead": "equals verify_tree on logits that are bf16 "
    "values already (no rounding ties); a uniform between the two roundings' "
    "acceptance ratios is a rounding tie, one outside is not",
    "residual inverse-CDF at large V": "equal to the draw in exact integer "
    "arithmetic (weights scaled by a common power of two, 24-bit dyadic "
    "uniforms) on residual rows at V = 128256, wherever no near tie is "
    "reported",
}
