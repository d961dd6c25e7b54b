// Host-side launchers of the verification kernels (internal to the library;
// the public surface is include/specverify.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/specverify.h"

namespace sv {

// Per-row argmax partial: value (NaN read as -inf) and lowest index.
struct ArgPart {
  float v;
  int32_t i;
};

// Elements per argmax work item (one CTA reduces one chunk of one row).
constexpr int kArgChunk = 16384;
inline int arg_splits(int V) { return (V + kArgChunk - 1) / kArgChunk; }

// Geometry of a verification call: rows are tree rows (chain: K+1 rows with
// a linear parent array).
struct VerifyShape {
  int B, n;      // n = K (chain) or N (tree): drafted tokens per sequence
  int R;         // draft rows per sequence
  int V;
  bool chain;
  int64_t rows() const { return (int64_t)B * (n + 1); }
};

// Device pointers of one verification call.
struct VerifyArgs {
  const void* target;
  const void* draft;
  const int32_t* q_row;        // tree only
  const int32_t* node_tokens;  // chain: draft_tokens [B,K]; tree: [B,N]
  const int32_t* parent;       // tree only
  int dt_target, dt_draft;
  spec_params_t prm;
  // outputs
  int32_t* count;       // accepted [B] / path_len [B]
  int32_t* path_nodes;  // tree only
  int32_t* out_tokens;  // [B, n+1]
  float* mass;          // chain [B,K]; tree [B,N+1]
  // workspace pieces
  uint32_t* status;
  int32_t* row_child;   // [rows] accepted child per row (-1 none)
  int32_t* row_token;   // [rows] sampled / argmax token per row
  ArgPart* arg_part;    // [rows * arg_splits(V)] (greedy)
};

// Event pair around a dominant kernel launch (no-op unless profiling is on).
void prof_begin(int kind, cudaStream_t st);
void prof_end(int kind, cudaStream_t st);

cudaError_t launch_greedy(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st);
cudaError_t launch_sampled(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st);
cudaError_t launch_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask,
                             uint64_t* bits, cudaStream_t st);
cudaError_t launch_philox(uint64_t seed, uint32_t offset, const int32_t* b, const int32_t* i,
                          const int32_t* slot, int n, float* out, cudaStream_t st);

// EAGLE-2 expand + rerank
struct Eagle2Cand {
  int32_t token;
  float logq;
};
cudaError_t launch_eagle2(const void* draft, int B, int V, int dtype, int depth, int topk,
                          int width, int total, float temperature, int32_t* node_tokens,
                          int32_t* parent, int32_t* q_row, float* value, uint8_t* mask,
                          Eagle2Cand* cand, uint32_t* status, cudaStream_t st);

}  // namespace sv
