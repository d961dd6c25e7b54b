// extern "C" entry points of libspecverify.so: host-side argument checks,
// workspace layout and dispatch to the kernels.  See include/specverify.h for
// the contract of every function.
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace of a verification call: [status | row_child | row_token | argmax parts]
struct VerifyWs {
  size_t off_child, off_token, off_parts, off_alpha, off_meta, off_qres;
  size_t off_tidx, off_tval, off_tcnt, off_out, off_qlist, total;
};
VerifyWs verify_ws(int B, int n, int V, bool chain) {
  const size_t rows = (size_t)B * (n + 1);
  VerifyWs w;
  w.off_child = kAlign;
  w.off_token = w.off_child + up(rows * sizeof(int32_t));
  w.off_parts = w.off_token + up(rows * sizeof(int32_t));
  w.off_alpha = w.off_parts + up(rows * (size_t)arg_splits(V) * sizeof(ArgPart));
  w.off_meta = w.off_alpha + up(rows * kAlphaSlots * sizeof(float));
  w.off_qres = w.off_meta + up(rows * (size_t)meta_rec_bytes(chain));
  w.off_tidx = w.off_qres + up(rows * sizeof(int32_t));
  w.off_tval = w.off_tidx + up(2 * rows * SPEC_MAX_TOP_K * sizeof(int32_t));
  w.off_tcnt = w.off_tval + up(2 * rows * SPEC_MAX_TOP_K * sizeof(float));
  w.off_out = w.off_tcnt + up(2 * rows * sizeof(int32_t));
  w.off_qlist = w.off_out + up(rows * sizeof(RowOut));
  w.total = w.off_qlist + up(rows * sizeof(int32_t));
  return w;
}
struct Eagle2Ws {
  size_t off_cand, total;
};
Eagle2Ws eagle2_ws(int B, int R) {
  Eagle2Ws w;
  w.off_cand = kAlign;
  w.total = w.off_cand + up((size_t)B * R * SPEC_EAGLE2_MAX_TOPK * sizeof(Eagle2Cand));
  return w;
}

bool dtype_ok(int d) { return d == SPEC_F32 || d == SPEC_BF16; }

int check_params(const spec_params_t* prm, int V, uint32_t allowed_flags = 0) {
  if (!prm) return SPEC_ERR_ARG;
  if (!(prm->temperature >= 0.f) || !std::isfinite(prm->temperature)) return SPEC_ERR_ARG;
  if ((prm->flags & ~allowed_flags) != 0) return SPEC_ERR_ARG;
  if (prm->draft_kind != SPEC_DRAFT_LOGITS && prm->draft_kind != SPEC_DRAFT_PROBS) return SPEC_ERR_DTYPE;
  if (prm->top_k < 0) return SPEC_ERR_ARG;
  if (!(prm->top_p > 0.f && prm->top_p <= 1.f)) return SPEC_ERR_ARG;
  if (prm->temperature > 0.f) {
    // a truncating transform runs on candidate lists of k_eff tokens
    const int keff = truncation_k(prm, V);
    if (keff > SPEC_MAX_TOP_K) return SPEC_ERR_UNSUPPORTED;
  }
  return SPEC_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

// Workspace of the LM head: [status | per-tile statistics [M, V/256] float2]
size_t lmhead_ws(int M, int V) {
  return kAlign + up((size_t)M * lmhead_tiles_n(V) * 2 * sizeof(float));
}
// Tree verification through the LM head: [verify | logits | stats | lse]
struct TreeLmWs {
  size_t off_logits, off_stats, off_lse, total;
};
TreeLmWs tree_lm_ws(int B, int N, int V) {
  const size_t rows = (size_t)B * (N + 1);
  TreeLmWs w;
  w.off_logits = verify_ws(B, N, V, false).total;
  w.off_stats = w.off_logits + up(rows * (size_t)V * 2);
  w.off_lse = w.off_stats + up(rows * lmhead_tiles_n(V) * 2 * sizeof(float));
  w.total = w.off_lse + up(rows * sizeof(float));
  return w;
}

// Points the call's scratch pieces into the caller's workspace.
int bind_verify_ws(const VerifyShape& s, VerifyArgs& a, void* ws, size_t ws_bytes) {
  const VerifyWs w = verify_ws(s.B, s.n, s.V, s.chain);
  if (!ws || ((uintptr_t)ws % kAlign) != 0) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < w.total) return SPEC_ERR_WORKSPACE;
  char* base = (char*)ws;
  a.status = (uint32_t*)base;
  a.row_child = (int32_t*)(base + w.off_child);
  a.row_token = (int32_t*)(base + w.off_token);
  a.arg_part = (ArgPart*)(base + w.off_parts);
  a.alpha_part = (float*)(base + w.off_alpha);
  a.meta = (unsigned char*)(base + w.off_meta);
  a.qres = (int32_t*)(base + w.off_qres);
  a.topk_idx = (int32_t*)(base + w.off_tidx);
  a.topk_val = (float*)(base + w.off_tval);
  a.topk_cnt = (int32_t*)(base + w.off_tcnt);
  a.rowout = (RowOut*)(base + w.off_out);
  a.qlist = (int32_t*)(base + w.off_qlist);
  a.qcount = (int32_t*)(base + 4);  // beside the status word, zeroed with it
  return SPEC_OK;
}

// Launches of a bound verification call (status word already cleared).
int launch_verify(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st) {
  if (s.B == 0) return SPEC_OK;
  if (a.prm.temperature == 0.f) return cuda_rc(launch_greedy(s, a, st));
  return cuda_rc(launch_sampled(s, a, st));
}

int run_verify(const VerifyShape& s, VerifyArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  int rc = bind_verify_ws(s, a, ws, ws_bytes);
  if (rc != SPEC_OK) return rc;
  if (a.prm.temperature != 0.f && !sampled_supported(s, a)) return SPEC_ERR_UNSUPPORTED;
  if (!(a.prm.temperature != 0.f && chain_small_writes_status(s, a))) {
    cudaError_t e = cudaMemsetAsync(a.status, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return launch_verify(s, a, st);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_workspace_bytes(int op, int B, int n, int V) {
  if (B < 0 || n < 0 || V < 1 || V > SPEC_MAX_VOCAB) return 0;
  if (op == SPEC_OP_CHAIN || op == SPEC_OP_TREE) {
    if (n > SPEC_MAX_TREE_NODES) return 0;
    return verify_ws(B, n, V, op == SPEC_OP_CHAIN).total;
  }
  if (op == SPEC_OP_EAGLE2) return eagle2_ws(B, n).total;
  if (op == SPEC_OP_LMHEAD) return n == 0 ? lmhead_ws(B, V) : 0;
  if (op == SPEC_OP_TREE_LMHEAD) {
    if (n > SPEC_MAX_TREE_NODES) return 0;
    return tree_lm_ws(B, n, V).total;
  }
  return 0;
}

int spec_verify_chain(const void* target_logits, const void* draft, const int32_t* draft_tokens,
                      int B, int K, int V, int dtype_target, int dtype_draft,
                      const spec_params_t* prm, int32_t* accepted, int32_t* out_tokens,
                      float* accept_mass, void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_SHAPE;
  if (V > SPEC_MAX_VOCAB || K > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  int rc = check_params(prm, V);
  if (rc != SPEC_OK) return rc;
  if (prm->draft_lse) return SPEC_ERR_ARG;
  if (!dtype_ok(dtype_target)) return SPEC_ERR_DTYPE;
  const bool greedy = prm->temperature == 0.f;
  if (!greedy && K > 0 && !dtype_ok(dtype_draft)) return SPEC_ERR_DTYPE;
  if (B > 0) {
    if (!target_logits || !accepted || !out_tokens) return SPEC_ERR_ARG;
    if (K > 0 && (!draft_tokens || !accept_mass)) return SPEC_ERR_ARG;
    if (!greedy && K > 0 && !draft) return SPEC_ERR_ARG;
  }
  VerifyShape s{B, K, K, V, true};
  VerifyArgs a{};
  a.target = target_logits;
  a.draft = greedy ? nullptr : draft;
  a.node_tokens = draft_tokens;
  a.dt_target = dtype_target;
  a.dt_draft = dtype_ok(dtype_draft) ? dtype_draft : SPEC_F32;
  a.prm = *prm;
  a.count = accepted;
  a.out_tokens = out_tokens;
  a.mass = accept_mass;
  return run_verify(s, a, workspace, ws_bytes, (cudaStream_t)stream);
}

int spec_verify_tree(const void* target_logits, const void* draft, const int32_t* q_row,
                     const int32_t* node_tokens, const int32_t* parent, int B, int N, int R,
                     int V, int dtype_target, int dtype_draft, const spec_params_t* prm,
                     int32_t* path_len, int32_t* path_nodes, int32_t* out_tokens,
                     float* accept_mass, void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || N < 0 || V < 1 || R < 0) return SPEC_ERR_SHAPE;
  if (V > SPEC_MAX_VOCAB || N > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  int rc = check_params(prm, V);
  if (rc != SPEC_OK) return rc;
  // given draft normalisers stand for softmax(z / T) of logit rows only
  if (prm->draft_lse && prm->temperature > 0.f &&
      (prm->draft_kind != SPEC_DRAFT_LOGITS || truncation_k(prm, V) > 0))
    return SPEC_ERR_ARG;
  if (!dtype_ok(dtype_target)) return SPEC_ERR_DTYPE;
  const bool greedy = prm->temperature == 0.f;
  if (!greedy && R > 0 && !dtype_ok(dtype_draft)) return SPEC_ERR_DTYPE;
  if (B > 0) {
    if (!target_logits || !path_len || !out_tokens || !accept_mass) return SPEC_ERR_ARG;
    if (N > 0 && (!node_tokens || !parent || !path_nodes)) return SPEC_ERR_ARG;
    if (!greedy && (!q_row || (R > 0 && !draft))) return SPEC_ERR_ARG;
  }
  VerifyShape s{B, N, R, V, false};
  VerifyArgs a{};
  a.target = target_logits;
  a.draft = greedy ? nullptr : draft;
  a.q_row = greedy ? nullptr : q_row;
  a.node_tokens = node_tokens;
  a.parent = parent;
  a.dt_target = dtype_target;
  a.dt_draft = dtype_ok(dtype_draft) ? dtype_draft : SPEC_F32;
  a.prm = *prm;
  if (greedy) a.prm.draft_lse = nullptr;
  a.count = path_len;
  a.path_nodes = path_nodes;
  a.out_tokens = out_tokens;
  a.mass = accept_mass;
  return run_verify(s, a, workspace, ws_bytes, (cudaStream_t)stream);
}

int spec_lm_head(const void* hidden, const void* w_vocab, int M, int H, int V, float temperature,
                 void* logits, float* row_lse, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || H < 1 || V < 1 || V > SPEC_MAX_VOCAB) return SPEC_ERR_SHAPE;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  if (row_lse && !(temperature > 0.f)) return SPEC_ERR_ARG;
  if (M > 0 && (!hidden || !w_vocab || !logits)) return SPEC_ERR_ARG;
  if (M > 0 && !lmhead_supported(hidden, w_vocab, H)) return SPEC_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || ws_bytes < lmhead_ws(M, V))
    return SPEC_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t* status = (uint32_t*)workspace;
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (M == 0) return SPEC_OK;
  float2* stats = row_lse ? (float2*)((char*)workspace + kAlign) : nullptr;
  return cuda_rc(launch_lmhead(hidden, w_vocab, M, H, V, temperature, (uint16_t*)logits, V, stats,
                               row_lse, status, st));
}

int spec_verify_tree_lmhead(const void* hidden, const void* w_vocab, int H, const void* draft,
                            const int32_t* q_row, const int32_t* node_tokens,
                            const int32_t* parent, int B, int N, int R, int V, int dtype_draft,
                            const spec_params_t* prm, int32_t* path_len, int32_t* path_nodes,
                            int32_t* out_tokens, float* accept_mass, void* logits,
                            void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || N < 0 || V < 1 || R < 0 || H < 1) return SPEC_ERR_SHAPE;
  if (V > SPEC_MAX_VOCAB || N > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  int rc = check_params(prm, V, SPEC_FLAG_TEST_STALL);
  if (rc != SPEC_OK) return rc;
  if (prm->draft_lse && prm->temperature > 0.f &&
      (prm->draft_kind != SPEC_DRAFT_LOGITS || truncation_k(prm, V) > 0))
    return SPEC_ERR_ARG;
  const bool greedy = prm->temperature == 0.f;
  if (!greedy && R > 0 && !dtype_ok(dtype_draft)) return SPEC_ERR_DTYPE;
  if (B > 0) {
    if (!hidden || !w_vocab || !path_len || !out_tokens || !accept_mass) return SPEC_ERR_ARG;
    if (N > 0 && (!node_tokens || !parent || !path_nodes)) return SPEC_ERR_ARG;
    if (!greedy && (!q_row || (R > 0 && !draft))) return SPEC_ERR_ARG;
    if (!lmhead_supported(hidden, w_vocab, H)) return SPEC_ERR_UNSUPPORTED;
  }
  const TreeLmWs lw = tree_lm_ws(B, N, V);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || ws_bytes < lw.total)
    return SPEC_ERR_WORKSPACE;
  char* base = (char*)workspace;
  uint16_t* lg = logits ? (uint16_t*)logits : (uint16_t*)(base + lw.off_logits);
  VerifyShape s{B, N, R, V, false};
  VerifyArgs a{};
  a.target = lg;
  a.draft = greedy ? nullptr : draft;
  a.q_row = greedy ? nullptr : q_row;
  a.node_tokens = node_tokens;
  a.parent = parent;
  a.dt_target = SPEC_BF16;
  a.dt_draft = dtype_ok(dtype_draft) ? dtype_draft : SPEC_F32;
  a.prm = *prm;
  if (greedy) a.prm.draft_lse = nullptr;
  a.count = path_len;
  a.path_nodes = path_nodes;
  a.out_tokens = out_tokens;
  a.mass = accept_mass;
  // the epilogue's normalisers serve the full-vocabulary sampled path
  const bool stats = !greedy && truncation_k(prm, V) == 0;
  a.tlse = stats ? (const float*)(base + lw.off_lse) : nullptr;
  rc = bind_verify_ws(s, a, workspace, ws_bytes);
  if (rc != SPEC_OK) return rc;
  if (!greedy && !sampled_supported(s, a)) return SPEC_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(a.status, 0, 2 * sizeof(uint32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
  const int M = B * (N + 1);
  rc = cuda_rc(launch_lmhead(hidden, w_vocab, M, H, V, prm->temperature, lg, V,
                             stats ? (float2*)(base + lw.off_stats) : nullptr,
                             stats ? (float*)(base + lw.off_lse) : nullptr, a.status, st,
                             (prm->flags & SPEC_FLAG_TEST_STALL) != 0));
  if (rc != SPEC_OK) return rc;
  return launch_verify(s, a, st);
}

int spec_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask, uint64_t* mask_bits,
                   void* stream) {
  if (B < 0 || N < 0 || N > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  if (mask_bits && N > 64) return SPEC_ERR_SHAPE;
  if (B > 0 && N > 0 && (!parent || (!mask && !mask_bits))) return SPEC_ERR_ARG;
  return cuda_rc(launch_tree_mask(parent, B, N, mask, mask_bits, (cudaStream_t)stream));
}

int spec_eagle2_expand_rerank(const void* draft_logits, int B, int V, int dtype, int depth,
                              int topk, int width, int total, const spec_params_t* prm,
                              int32_t* node_tokens, int32_t* parent, int32_t* q_row,
                              float* value, uint8_t* mask, void* workspace, size_t ws_bytes,
                              void* stream) {
  if (B < 0 || V < 1 || V > SPEC_MAX_VOCAB) return SPEC_ERR_SHAPE;
  if (depth < 1 || topk < 1 || topk > SPEC_EAGLE2_MAX_TOPK || topk > V || width < 1)
    return SPEC_ERR_SHAPE;
  if (total < 1 || total > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  // candidates: topk at layer 1, then min(width, layer size) * topk per layer
  int64_t ncand = 0, layer = topk;
  for (int d = 1; d <= depth; ++d) {
    ncand += layer;
    layer = (int64_t)(layer < width ? layer : width) * topk;
  }
  if (total > ncand || ncand > SPEC_EAGLE2_MAX_CANDIDATES) return SPEC_ERR_SHAPE;
  if (width > SPEC_EAGLE2_MAX_WIDTH) return SPEC_ERR_SHAPE;
  if (!prm || !(prm->temperature > 0.f) || !std::isfinite(prm->temperature)) return SPEC_ERR_ARG;
  if (!dtype_ok(dtype)) return SPEC_ERR_DTYPE;
  const int R = 1 + (depth - 1) * width;
  if (B > 0 && (!draft_logits || !node_tokens || !parent || !q_row || !value)) return SPEC_ERR_ARG;
  const Eagle2Ws w = eagle2_ws(B, R);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || ws_bytes < w.total)
    return SPEC_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t* status = (uint32_t*)workspace;
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
  return cuda_rc(launch_eagle2(draft_logits, B, V, dtype, depth, topk, width, total,
                               prm->temperature, node_tokens, parent, q_row, value, mask,
                               prm->draft_lse,
                               (Eagle2Cand*)((char*)workspace + w.off_cand), status, st));
}

int spec_get_status(const void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return SPEC_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_philox_uniforms(uint64_t seed, uint32_t offset, const int32_t* b, const int32_t* idx,
                         const int32_t* slot, int n, float* out, void* stream) {
  if (n < 0) return SPEC_ERR_SHAPE;
  if (n > 0 && (!b || !idx || !slot || !out)) return SPEC_ERR_ARG;
  return cuda_rc(launch_philox(seed, offset, b, idx, slot, n, out, (cudaStream_t)stream));
}

const char* spec_error_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument";
    case SPEC_ERR_DTYPE: return "unsupported dtype or draft kind";
    case SPEC_ERR_SHAPE: return "invalid or unsupported sizes";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_UNSUPPORTED: return "unsupported parameter combination";
    default: return "unknown error";
  }
}

}  // extern "C"
