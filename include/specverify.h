/*
 * specverify.h -- C ABI of the GB300 speculative-decoding verification
 * library (libspecverify.so, sm_103a).
 *
 * What it computes.  Given target-model logits at every drafted position and
 * the draft model's distributions, decide which drafted tokens a target
 * sampler would have produced, exactly as sampling from the target would:
 *
 *   accept drafted x with probability min(1, p(x)/q(x)), left to right, stop
 *   at the first rejection and draw the replacement from norm(max(0, p - q));
 *   if every draft is accepted draw a bonus token from p at the last row.
 *
 * (exactness rule of "投机解码与 EAGLE"; a(x) and r(x), section 二 of
 * "064 · 投机解码：小模型先起草，大模型怎样并行验收而不改变分布"; §2.1 of the
 * EAGLE-2 notes.)  p and q are taken after the same temperature / top-k /
 * top-p transform ("064 · 投机解码", section 二).  Temperature 0 selects the
 * greedy rule (accept while the draft equals the target argmax, then emit the
 * argmax; "贪婪情形简化" of "投机解码与 EAGLE").  Trees follow the EAGLE
 * description (a rejected token lets the other branches be tried, EAGLE-2
 * notes §2.2) and EAGLE-2's expand / rerank (§4.1-4.2).
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers owned by the caller, row-major
 *     and contiguous (last dimension fastest).  The library allocates nothing
 *     and keeps no pointer after the call.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*, NULL =
 *     legacy default stream); calls return as soon as the work is enqueued.
 *     Outputs and the workspace must not be touched by other work on other
 *     streams until the enqueued work has finished.
 *   - Logit dtypes: SPEC_F32 (float32) or SPEC_BF16 (bfloat16 stored as
 *     uint16).  Token and index arrays are int32.
 *   - Return value: SPEC_OK or a negative SPEC_ERR_* code.  Argument errors
 *     are detected on the host before anything is enqueued.  Data-dependent
 *     conditions found on the device (NaN logits, a drafted token with
 *     q(x) = 0, ...) never stop a kernel: they set bits of a status word kept
 *     in the workspace, read back with spec_get_status().
 *   - Random numbers: one uniform per decision from Philox4x32-10 (Salmon et
 *     al., SC'11) with key = (seed low 32 bits, seed high 32 bits) and counter
 *     (b, i, slot, philox_offset); u = (word0 >> 8) * 2^-24.  slot 0: accept
 *     test of drafted token i; slot 1: replacement / bonus draw at target
 *     row i.  The draw used for a decision does not depend on other outcomes.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
#define SPEC_OK 0
#define SPEC_ERR_ARG (-1)         /* NULL pointer, negative size, bad param */
#define SPEC_ERR_DTYPE (-2)       /* unknown dtype or draft kind           */
#define SPEC_ERR_SHAPE (-3)       /* sizes inconsistent or over the limits */
#define SPEC_ERR_CUDA (-4)        /* a CUDA runtime call failed            */
#define SPEC_ERR_WORKSPACE (-5)   /* workspace NULL, misaligned or small   */
#define SPEC_ERR_UNSUPPORTED (-6) /* valid request this build cannot serve */

/* ---- dtypes and draft kinds ---- */
#define SPEC_F32 0
#define SPEC_BF16 1
#define SPEC_DRAFT_LOGITS 0 /* draft rows are logits: q = softmax(z / T)  */
#define SPEC_DRAFT_PROBS 1  /* draft rows are probabilities: z = log q    */

/* ---- limits ---- */
#define SPEC_MAX_VOCAB (1 << 24)  /* V                                     */
#define SPEC_MAX_TOP_K 128        /* tokens a truncating transform keeps   */
#define SPEC_MAX_CHILDREN 64      /* children of one tree node             */
#define SPEC_MAX_TREE_NODES 1024  /* N (tree) and K (chain)                */
#define SPEC_EAGLE2_MAX_TOPK 32   /* children per expanded EAGLE-2 node    */
#define SPEC_EAGLE2_MAX_WIDTH 2048 /* nodes kept per EAGLE-2 layer          */
#define SPEC_EAGLE2_MAX_CANDIDATES 4096 /* EAGLE-2 candidates per sequence */

/* ---- device status bits (spec_get_status) ---- */
#define SPEC_STATUS_NAN 1u            /* a logit row had NaN / no finite value */
#define SPEC_STATUS_QZERO_ACCEPT 2u   /* drafted token with q(x) = 0 accepted  */
#define SPEC_STATUS_RESIDUAL_ZERO 4u  /* residual had no mass; drew from p     */
#define SPEC_STATUS_DRAFT_EXHAUSTED 8u /* siblings' tokens held all of q       */
#define SPEC_STATUS_CDF_FALLBACK 16u  /* rounding: inverse CDF took last token */
#define SPEC_STATUS_BAD_TREE 32u      /* parent / q_row entry out of range     */
#define SPEC_STATUS_TOKEN_RANGE 64u   /* drafted token outside [0, V): reject  */
#define SPEC_STATUS_TIMEOUT 128u      /* a bounded device wait gave up         */

/* ---- operations for spec_workspace_bytes ---- */
#define SPEC_OP_CHAIN 1
#define SPEC_OP_TREE 2
#define SPEC_OP_EAGLE2 3
#define SPEC_OP_LMHEAD 4       /* spec_lm_head: B = rows M, n = 0           */
#define SPEC_OP_TREE_LMHEAD 5  /* spec_verify_tree_lmhead: n = N            */

/* Test-only flag of spec_verify_tree_lmhead (SPEC_ERR_ARG elsewhere): the
   LM-head kernel's copy producer withholds the first shared-memory stage, so
   that the tensor-core issuer's bounded wait on it gives up (after about a
   second), SPEC_STATUS_TIMEOUT is set and the call still completes.  It
   exercises the failure path of the device waits without faulting anything;
   the outputs of such a call are meaningless. */
#define SPEC_FLAG_TEST_STALL 0x80000000u

/* Sampling parameters (plain data, 40 bytes). */
typedef struct spec_params {
  float temperature;      /* > 0: sampling rule; == 0: greedy argmax rule  */
  int32_t top_k;          /* 0 = off; keeps min(top_k, V) tokens           */
  float top_p;            /* in (0, 1]; 1 = off                            */
  /* With top-k or top-p the kept set min(top_k, V) (V when top_k = 0) must
     hold at most SPEC_MAX_TOP_K tokens, else SPEC_ERR_UNSUPPORTED. */
  int32_t draft_kind;     /* SPEC_DRAFT_LOGITS or SPEC_DRAFT_PROBS         */
  uint64_t seed;          /* Philox key                                    */
  uint32_t philox_offset; /* fourth Philox counter word                    */
  uint32_t flags;         /* 0, or SPEC_FLAG_TEST_STALL (tests only)       */
  /* Optional device array [B, R] float32 (NULL = unused): the log2
     normaliser log2 sum_v 2^(z_v log2(e) / temperature) of each draft row.
     spec_eagle2_expand_rerank writes it (the expand already sums every
     draft row); spec_verify_tree then reads it instead of summing the draft
     rows again, which is valid only for logit drafts at the same
     temperature, without top-k / top-p (else SPEC_ERR_ARG; ignored at
     temperature 0).  Must be NULL for spec_verify_chain. */
  float* draft_lse;
} spec_params_t;

/*
 * Workspace size in bytes for one call of `op` (SPEC_OP_CHAIN with n = K,
 * SPEC_OP_TREE with n = N, SPEC_OP_EAGLE2 with n = number of draft rows per
 * sequence, SPEC_OP_LMHEAD with B = rows and n = 0, SPEC_OP_TREE_LMHEAD
 * with n = N).  The workspace must be 256-byte aligned device memory; its
 * contents need no initialisation and are overwritten by every call.  Returns
 * 0 for invalid sizes.
 */
size_t spec_workspace_bytes(int op, int B, int n, int V);

/*
 * Chain verification (the listing of "064 · 投机解码", section 三; steps 3-4 of
 * "投机解码与 EAGLE").
 *
 * target_logits [B, K+1, V] dtype_target: target logits at the K drafted
 *     positions and the bonus position.
 * draft [B, K, V] dtype_draft: draft logits or probabilities
 *     (prm->draft_kind).  Not read, and may be NULL, when temperature == 0.
 * draft_tokens [B, K] int32: the drafted tokens x_0 .. x_{K-1}.
 * accepted [B] int32 (out): number n of accepted drafts, 0 .. K.
 * out_tokens [B, K+1] int32 (out): x_0 .. x_{n-1}, then the replacement
 *     (n < K) or bonus (n == K) token, then -1 padding.
 * accept_mass [B, K] float32 (out): alpha_k = sum_x min(p_k(x), q_k(x)) for
 *     every k (also after the first rejection); at temperature 0 the
 *     indicator 1[x_k == argmax_k].
 * B >= 0 (0 = nothing to do), 0 <= K <= SPEC_MAX_TREE_NODES,
 * 1 <= V <= SPEC_MAX_VOCAB.  Sampling over the full vocabulary streams rows
 * whose pointers are 16-byte aligned with V % 8 == 0 up to V = 524288; other
 * rows (odd lengths, unaligned pointers) up to about 200 K float32 or 400 K
 * bfloat16 logits per row pair; beyond that the call returns
 * SPEC_ERR_UNSUPPORTED before launching anything.  The same holds for
 * spec_verify_tree.
 */
int spec_verify_chain(const void* target_logits, const void* draft,
                      const int32_t* draft_tokens, int B, int K, int V,
                      int dtype_target, int dtype_draft,
                      const spec_params_t* prm, int32_t* accepted,
                      int32_t* out_tokens, float* accept_mass,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Tree verification (EAGLE static or dynamic trees; EAGLE-2 notes §2.2 and
 * §4.2; "EAGLE:树形草稿" of "投机解码与 EAGLE").
 *
 * Drafted nodes j = 0 .. N-1; parent[b, j] = -1 for a child of the root, else
 * an index in [0, j) (parents precede children).  Tree row r = 0 is the root
 * position, row r = j + 1 the position after node j.
 *
 * target_logits [B, N+1, V]: target logits per tree row.
 * draft [B, R, V]: draft rows; q_row [B, N+1] int32 names the draft row of
 *     each tree row (-1 = none; required for rows that have children).  Not
 *     read when temperature == 0 (draft and q_row may then be NULL).
 * node_tokens [B, N], parent [B, N] int32.
 * At each row the children are tried in index order: accept child c with
 * token x iff u(b, c, 0) < p'(x)/q'(x); on rejection p' <- norm(max(0,
 * p' - q')) and x leaves q' (siblings are drafted without replacement); if
 * no child is accepted the emitted token is drawn from p' with u(b, r, 1)
 * (a leaf: bonus from p).  The walk follows accepted children from the root.
 * path_len [B] (out): accepted drafted nodes on the path.
 * path_nodes [B, N] (out): their node indices, -1 padded.
 * out_tokens [B, N+1] (out): their tokens, then the sampled token, -1 padded.
 * accept_mass [B, N+1] float32 (out): alpha per tree row (NaN where the row
 *     has no draft row; at temperature 0: 1 if a child matches the argmax,
 *     0 if none does, NaN for a row without children).
 * prm->draft_lse (optional, [B, R]): the draft rows' log2 normalisers, as
 *     spec_eagle2_expand_rerank writes them; the caller vouches that they
 *     belong to these rows at this temperature.
 */
int spec_verify_tree(const void* target_logits, const void* draft,
                     const int32_t* q_row, const int32_t* node_tokens,
                     const int32_t* parent, int B, int N, int R, int V,
                     int dtype_target, int dtype_draft,
                     const spec_params_t* prm, int32_t* path_len,
                     int32_t* path_nodes, int32_t* out_tokens,
                     float* accept_mass, void* workspace, size_t ws_bytes,
                     void* stream);

/*
 * Target LM head of the verification pass (step 2 of the draft/verify loop
 * of "投机解码与 EAGLE": one target forward over every drafted position; its
 * last layer maps each position's final hidden state to logits).
 *
 * logits [M, V] bf16 (out) = hidden [M, H] bf16 x w_vocab^T, w_vocab [V, H]
 *     bf16 (row-major, the layout of a linear layer's weight); products
 *     accumulated in float32 on the tensor cores, rounded to bf16 (nearest,
 *     ties to even).
 * row_lse [M] float32 (out, may be NULL; needs temperature > 0): each row's
 *     base-2 log normaliser log2 sum_v 2^(z_v log2(e) / temperature) of the
 *     rounded logits, the first pass of verification taken in the GEMM's
 *     epilogue.
 * Requirements: H % 8 == 0 (rows of 16-byte multiples), hidden and w_vocab
 * 16-byte aligned, else SPEC_ERR_UNSUPPORTED; M >= 0, 1 <= V <=
 * SPEC_MAX_VOCAB.  Workspace: spec_workspace_bytes(SPEC_OP_LMHEAD, M, 0, V)
 * (status word and per-tile statistics).  Status bits (SPEC_STATUS_TIMEOUT)
 * via spec_get_status.
 */
int spec_lm_head(const void* hidden, const void* w_vocab, int M, int H, int V,
                 float temperature, void* logits, float* row_lse,
                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Tree verification with the target logits computed from the target's final
 * hidden states by the LM head (spec_lm_head followed by spec_verify_tree,
 * with the target rows' normalisers taken in the GEMM's epilogue so that
 * verification reads each target row once).
 *
 * hidden [B, N+1, H] bf16: the target's final hidden state at each tree row;
 * w_vocab [V, H] bf16; the other arguments as for spec_verify_tree (the
 * target logits are bf16).  logits [B, N+1, V] bf16 (out, may be NULL): the
 * computed target logits; NULL keeps them in the workspace.  Workspace:
 * spec_workspace_bytes(SPEC_OP_TREE_LMHEAD, B, N, V).  Requirements and
 * errors as for spec_lm_head and spec_verify_tree.
 */
int spec_verify_tree_lmhead(const void* hidden, const void* w_vocab, int H,
                            const void* draft, const int32_t* q_row,
                            const int32_t* node_tokens, const int32_t* parent,
                            int B, int N, int R, int V, int dtype_draft,
                            const spec_params_t* prm, int32_t* path_len,
                            int32_t* path_nodes, int32_t* out_tokens,
                            float* accept_mass, void* logits,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * Tree attention mask (EAGLE-2 notes §4.2: each token sees only its
 * ancestors; the chain case is the lower-triangular causal mask).
 * mask [B, N, N] uint8 (out): mask[b, i, j] = 1 iff j is i or an ancestor of
 *     i; the committed prefix is visible to every node and is not included.
 * mask_bits [B, N] uint64 (out, may be NULL; requires N <= 64): bit j of
 *     mask_bits[b, i] = mask[b, i, j].  Either output may be NULL, not both.
 * An out-of-range parent ends that node's ancestor walk.
 */
int spec_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask,
                   uint64_t* mask_bits, void* stream);

/*
 * EAGLE-2 dynamic tree: expand and rerank (EAGLE-2 notes §4.1-4.2).
 *
 * draft_logits [B, 1 + (depth-1)*width, V]: row 0 is the draft distribution
 *     at the root; row 1 + (d-1)*width + r is the one after the r-th kept node
 *     of layer d (the draft forward between layers is the caller's).
 * q = softmax(z / prm->temperature) (temperature > 0; top_k / top_p unused).
 * Layer 1 = the `topk` most probable tokens of row 0 (ties: lower index),
 * value = log q.  Layer d+1 = the `topk` best tokens of each kept node's row,
 * value = parent value + log q.  Each layer keeps its `width` best nodes by
 * (value desc, candidate id asc), id = (layer, parent rank, child rank).
 * All candidates of all layers are reranked by (value desc, depth asc, id
 * asc) and the best `total` kept, in that order (parents before children).
 * node_tokens [B, total], parent [B, total] (-1 = root child),
 * q_row [B, total+1] (draft row of each tree row or -1; row 0 -> 0),
 * value [B, total] float32 (sum of log q along the path),
 * mask [B, total, total] uint8 (may be NULL) as spec_tree_mask.
 * prm->draft_lse (optional out, [B, R] float32): each draft row's log2
 *     normaliser at this temperature, for spec_verify_tree.
 * Limits: 1 <= topk <= SPEC_EAGLE2_MAX_TOPK, width <= topk * width of the
 * layer above, total <= number of candidates, total <= SPEC_MAX_TREE_NODES.
 */
int spec_eagle2_expand_rerank(const void* draft_logits, int B, int V,
                              int dtype, int depth, int topk, int width,
                              int total, const spec_params_t* prm,
                              int32_t* node_tokens, int32_t* parent,
                              int32_t* q_row, float* value, uint8_t* mask,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Synchronously read the status word of the last call that used `workspace`
 * (waits for `stream`).  SPEC_STATUS_* bits; 0 = nothing to report.
 */
int spec_get_status(const void* workspace, uint32_t* status, void* stream);

/*
 * KV-cache commit after verification ("KV cache rollback" and step 4 of the
 * Vietnamese speculative-decoding page; "El baile de caché KV" of the
 * Spanish page).  The verification pass wrote the drafted positions' KV
 * entries after each sequence's committed prefix; this keeps those of the
 * accepted drafts, in path order, and sets the logical lengths.  The token
 * drawn after the path has no entry yet (the next forward pass writes it).
 *
 * Chain (path_nodes == NULL): the accepted drafts are the first path_len[b]
 *     positions after the prefix, already in place; nothing moves.
 * Tree: drafted node j's entry is at position prefix_len[b] + j; the path
 *     path_nodes[b, 0 .. path_len[b]) (node indices, strictly increasing, as
 *     spec_verify_tree returns them) moves to positions prefix_len[b] + i.
 *     The move runs in place in path order, which is safe because
 *     path_nodes[b, i] >= i.
 * new_len[b] (out) = prefix_len[b] + path_len[b], or -1 if the path is
 *     invalid (path_len outside [0, N], a node outside [0, N) or not above
 *     the previous one); such a sequence is left unchanged.
 * Positions past the new length keep whatever they held.
 *
 * Layout: the entry of sequence b at position s is, for every plane
 * (p1 < n1, p2 < n2), the row_bytes bytes at
 *     kv + b*stride_b + p1*stride_1 + p2*stride_2 + s*stride_pos   (bytes),
 * which describes head-major caches ([L*2, B, H, S, D]: n1 = 2L, n2 = H),
 * position-major ones ([B, S, L*2*H*D]: n1 = n2 = 1) and the like.  The
 * caller guarantees that the addressed rows of positions up to
 * prefix_len[b] + N lie in its allocation and do not overlap one another.
 * Device arrays: prefix_len [B], path_nodes [B, N] (or NULL), path_len [B],
 * new_len [B].  Errors: SPEC_ERR_SHAPE for negative sizes or a negative
 * stride; SPEC_ERR_ARG for a NULL prefix_len, path_len or new_len, or a NULL
 * kv for a tree (when B > 0; a chain does not touch kv).
 */
int spec_kv_commit(void* kv, int B, int n1, int n2, int64_t stride_b,
                   int64_t stride_1, int64_t stride_2, int64_t stride_pos,
                   int row_bytes, const int32_t* prefix_len,
                   const int32_t* path_nodes, const int32_t* path_len, int N,
                   int32_t* new_len, void* stream);

/*
 * Acceptance records over verification outcomes, accumulated across calls:
 * the distribution of the accepted length per round, not only its mean
 * ("064 · 投机解码", section 五), the acceptance rate of drafted tokens by
 * position in the draft tree and by depth (EAGLE-2 notes §3.1, Fig. 5), and
 * by interval of the draft model's confidence in its token (§3.2, Fig. 6).
 *
 * A round is one sequence's verification.  A drafted token is TESTED iff its
 * parent is the root or on the accepted path and no sibling with a lower node
 * index was accepted (the tree rule tries siblings in node order); it is
 * ACCEPTED iff it is on the path.  (When the draft distribution runs out of
 * mass the rule stops trying siblings early; the outcome does not show this
 * and such siblings count as tested.)  Depth: 1 for a child of the root,
 * else the parent's depth + 1.
 *
 * Chain (parent == path_nodes == NULL): count[b] = accepted drafts of
 *     spec_verify_chain; token k is tested iff k <= count[b], accepted iff
 *     k < count[b]; its depth is k + 1.
 * Tree: count[b] = path_len[b], path_nodes [B, n] and parent [B, n] as
 *     spec_verify_tree takes and returns them.
 * confidence [B, n] (float32, or NULL for no calibration record): the draft
 *     model's probability of each drafted token.  It is clamped to [0, 1] and
 *     counted in bin floor(c * nbins) (float32 product; 1.0 in the last bin);
 *     NaN is not binned.
 *
 * Records (device arrays owned by the caller, ADDED to, never cleared; any
 * pointer may be NULL to skip that record):
 *   len_hist [n + 1]     rounds by accepted length (chain count / path_len)
 *   node_tested [n], node_accepted [n]      by node index (chain: position)
 *   depth_tested [n], depth_accepted [n]    index = depth - 1
 *   calib_tested [nbins], calib_accepted [nbins], calib_conf_sum [nbins]
 *                        (double: sum of the clamped confidences)
 *   invalid [1]          rounds that are not a root path of their tree
 *                        (count outside [0, n], a path node out of range or
 *                        not a child of the previous one, a parent array
 *                        not pointing to earlier nodes); they add nothing
 *                        else.
 * Integer records are exact; calib_conf_sum is summed in double in no fixed
 * order.  Calls on one record that overlap on the GPU still add correctly
 * (device atomics).
 * Errors: SPEC_ERR_ARG for a NULL count or out, exactly one of parent /
 * path_nodes NULL, or (B > 0) an array not aligned to its element size (4
 * bytes for the inputs, 8 for the records); SPEC_ERR_SHAPE for B < 0, n
 * outside [1, SPEC_MAX_TREE_NODES], or nbins outside [1,
 * SPEC_STATS_MAX_BINS] when confidence is given.  B == 0 does nothing.
 */
#define SPEC_STATS_MAX_BINS 1024
typedef struct {
  int64_t* len_hist;
  int64_t* node_tested;
  int64_t* node_accepted;
  int64_t* depth_tested;
  int64_t* depth_accepted;
  int64_t* calib_tested;
  int64_t* calib_accepted;
  double* calib_conf_sum;
  int64_t* invalid;
} spec_accept_stats_t;
int spec_accept_stats(const int32_t* count, const int32_t* parent,
                      const int32_t* path_nodes, const float* confidence,
                      int B, int n, int nbins, const spec_accept_stats_t* out,
                      void* stream);

/*
 * Attention of the verification pass over a draft tree (EAGLE-2 notes §4.2:
 * the selected draft tokens are flattened and verified in one forward pass,
 * each seeing only the committed prefix, its ancestors and itself; the
 * Spanish lesson's Medusa section uses the same tree attention).  For
 * sequence b with prefix length P = prefix_len[b] and drafted node i:
 *
 *   o[b,i,h] = sum_s softmax_s(scale * q[b,i,h] . k[b,h/G,s]) v[b,h/G,s]
 *   over s < P, and s = P + j for every bit j set in mask_bits[b, i]
 *
 * (G = Hq / Hkv query heads per key/value head).  The drafted tokens' keys
 * and values are already in the cache at positions P .. P + N - 1 in node
 * order; mask_bits is spec_tree_mask's 64-bit output (bit j of row i:
 * j is an ancestor of i, or i itself).
 *
 * Layout (device, bf16 stored as uint16, row-major, contiguous):
 *   q [B, N, Hq, D], out [B, N, Hq, D] (written), k_cache and v_cache
 *   [B, Hkv, S, D], prefix_len [B] int32, mask_bits [B, N] uint64.
 * Softmax and accumulation in float32; the output is rounded to bf16.
 * prefix_len is clamped to [0, S - N].
 * Errors: SPEC_ERR_SHAPE unless 1 <= N <= 64, Hq % Hkv == 0, S >= N and
 * B, Hkv <= 65535;
 * SPEC_ERR_UNSUPPORTED unless D == 128, or when q or out is not 16-byte
 * aligned (rows are moved as 16-byte words); SPEC_ERR_ARG for scale <= 0 or
 * not finite, a NULL pointer (B > 0), caches not 16-byte aligned, q, out or
 * prefix_len not 4-byte aligned, or mask_bits not 8-byte aligned;
 * SPEC_ERR_SHAPE when B * Hkv * S reaches 2^31 cache rows; SPEC_ERR_CUDA if
 * the caches cannot be described to the copy engine.  B == 0 does nothing.
 * Runs on the tensor cores (tcgen05): one CTA per 256 query rows of one
 * (sequence, key/value head).
 */
int spec_tree_attention(const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* prefix_len,
                        const uint64_t* mask_bits, int B, int N, int Hq,
                        int Hkv, int D, int S, float scale, void* out,
                        void* stream);

/*
 * The uniforms the kernels draw: out[i] = u(b[i], idx[i], slot[i]) for the
 * given seed and offset (all arrays device, length n).  Lets callers and
 * tests check the device generator bit for bit.
 */
int spec_philox_uniforms(uint64_t seed, uint32_t offset, const int32_t* b,
                         const int32_t* idx, const int32_t* slot, int n,
                         float* out, void* stream);

/* Human-readable name of a return code. */
const char* spec_error_string(int code);

/*
 * Chain verification without a workspace, for callers that cannot allocate
 * device memory (an engine plugin handed only its input and output buffers,
 * or a decode loop where cudaMalloc is not allowed).  No counterpart on the
 * pages: for the calls it serves it computes what spec_verify_chain computes
 * (same arguments minus the workspace) and differs only in where its scratch
 * lives.  Not served: sampling with top-k / top-p truncation (temperature
 * > 0 with top_k > 0 or top_p < 1) and rows the streaming kernels cannot
 * take, both SPEC_ERR_UNSUPPORTED; given draft normalisers (draft_lse),
 * SPEC_ERR_ARG.  Its status bits are read with spec_get_status_noalloc.
 *
 * The scratch is one fixed array inside the library (about 1.7 MiB) that
 * every GPU which loads the library holds until the process exits.  The first
 * call on a device looks up that array's device address with the device
 * current, so make the first call before any stream capture.  All calls on a
 * device share the array and leave their contents in it: calls whose GPU work
 * overlaps (several streams or host threads on one device) race and must be
 * serialised by the caller.  Limits: B*(K+1) <= SPEC_NOALLOC_MAX_ROWS and
 * B*(K+1)*ceil(V/16384) <= SPEC_NOALLOC_MAX_PARTS; larger requests return
 * SPEC_ERR_SHAPE before any GPU work.  Allocates nothing.
 */
#define SPEC_NOALLOC_MAX_ROWS 8192
#define SPEC_NOALLOC_MAX_PARTS 65536
int spec_verify_chain_noalloc(const void* target_logits, const void* draft,
                              const int32_t* draft_tokens, int B, int K, int V,
                              int dtype_target, int dtype_draft,
                              const spec_params_t* prm, int32_t* accepted,
                              int32_t* out_tokens, float* accept_mass,
                              void* stream);

/*
 * Status bits (SPEC_STATUS_*) of the last spec_verify_chain_noalloc call on
 * the current device: copies the status word out of the library's fixed
 * array into the host word *status and waits for `stream`.  Like the call
 * itself it allocates nothing; SPEC_ERR_ARG if status is NULL.
 */
int spec_get_status_noalloc(uint32_t* status, void* stream);

/*
 * Kernel timing for benchmarks.  spec_profile_enable(1) clears the record and
 * makes every later call bracket its dominant kernel with a pair of CUDA
 * events recorded on the caller's stream (at most 16384 pairs); n > 1
 * brackets only every n-th launch of each kind (a sample, so that the
 * events' own cost stays off most calls); 0 turns it off; a negative n is
 * SPEC_ERR_ARG.  spec_profile_read waits for the recorded events and returns the total
 * milliseconds and number of launches of one kernel kind:
 *   SPEC_PROF_ARGMAX    greedy argmax streaming kernel,
 *   SPEC_PROF_VERIFY    sampled row-verification kernel,
 *   SPEC_PROF_EXPAND    EAGLE-2 draft-row top-k kernel,
 *   SPEC_PROF_KV        KV-cache commit move kernel,
 *   SPEC_PROF_STATS     acceptance-records kernel,
 *   SPEC_PROF_ATTN      tree-attention kernel,
 *   SPEC_PROF_LMHEAD    LM-head GEMM kernel.
 * Returns SPEC_ERR_SHAPE if pairs were dropped.  Not thread-safe.
 */
#define SPEC_PROF_ARGMAX 0
#define SPEC_PROF_VERIFY 1
#define SPEC_PROF_EXPAND 2
#define SPEC_PROF_KV 3
#define SPEC_PROF_STATS 4
#define SPEC_PROF_ATTN 5
#define SPEC_PROF_LMHEAD 6
int spec_profile_enable(int on);
int spec_profile_read(int kind, double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
