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
  __host__ __device__ int64_t rows() const { return (int64_t)B * (n + 1); }
};

// Outcome of a row's sibling recursion as far as the streaming verifier
// takes it (the walk finishes it for the rows on the accepted path).
//   child >= 0: that drafted child was accepted;
//   child == -1: every child was rejected (or a leaf): the row's token is
//     drawn from max(0, p - Cn q) (p when Cn = 0), or from max(0, p - Cc q)
//     (p when Cc = 0) if the former has no mass;
//   child == -2: child k was rejected and a later child needs the mass of
//     max(0, p - Cn q), which takes another pass over the row.
// Cc, W, D are the recursion state: current residual coefficient, its mass
// and the draft mass left.  Lp / Lq are the row's base-2 log normalisers
// (invZq = 1 / sum q for probability rows at T = 1).
struct RowOut {
  int child;
  int k;
  float Cc, W, D, Cn;
  float Lp, Lq, invZq;
  uint32_t bits;
  int pad[6];
};
static_assert(sizeof(RowOut) == 64, "row outcome layout");

// Device pointers of one verification call.
struct VerifyArgs {
  const void* target;
  const void* draft;
  const int32_t* q_row;        // tree only
  const int32_t* node_tokens;  // chain: draft_tokens [B,K]; tree: [B,N]
  const int32_t* parent;       // tree only
  const float* tlse;           // [rows] target rows' base-2 log normalisers
                               // at the call's temperature, or null (the
                               // streaming kernel then sums the rows itself)
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
  float* alpha_part;    // [rows * 8] per-CTA acceptance-mass partials
  unsigned char* meta;  // [rows * meta_rec_bytes(chain)] per-row records
  int32_t* qres;        // [rows] resolved draft row per tree row (-1 none)
  int32_t* topk_idx;    // [2 * rows * SPEC_MAX_TOP_K] top-k candidates
  float* topk_val;      //   (target rows, then draft rows)
  int32_t* topk_cnt;    // [2 * rows]
  RowOut* rowout;       // [rows] row outcomes of the streaming verifier
  int32_t* qlist;       // [rows] rows that have a draft row (the streaming kernel's work)
  int32_t* qcount;      //   their number (zeroed with the status word)
};

// Tokens a truncating sampling transform keeps per row: min(top_k, V), with
// top_k = 0 meaning V; 0 when neither top-k nor top-p truncates anything.
inline int truncation_k(const spec_params_t* p, int V) {
  const int k = (p->top_k <= 0 || p->top_k >= V) ? V : p->top_k;
  if (p->top_p >= 1.f && k == V) return 0;
  return k;
}

// Sampled verification with top-k / top-p truncation (k <= SPEC_MAX_TOP_K).
cudaError_t launch_sparse(const VerifyShape& s, const VerifyArgs& a, int k, cudaStream_t st);

// Per-row record of the pipelined kernel: a 16-byte header, 16 bytes per
// child slot and 4 bytes of accept uniform per slot, padded to 16 bytes (one
// slot for a chain, SPEC_MAX_CHILDREN for a tree).
inline int meta_kidcap(bool chain) { return chain ? 1 : SPEC_MAX_CHILDREN; }
inline int meta_rec_bytes(bool chain) {
  return (16 + 20 * meta_kidcap(chain) + 15) / 16 * 16;
}

// Per-row slots of alpha partials (one per CTA of a cluster of up to 8).
constexpr int kAlphaSlots = 8;

// Launch parameters of the streaming sampled-verification kernel.
struct StreamParams {
  VerifyShape s;
  VerifyArgs a;
  int C;          // CTAs per cluster (vocabulary slices per row)
  int slice;      // vocabulary elements per CTA (multiple of 8)
  int nch;        // 4096-element chunks per slice
  int stages;     // shared-memory ring stages
  int nclusters;  // persistent clusters (set by the launcher)
  int qk;         // draft kind: 0 logits, 1 probabilities at T = 1, 2 probabilities
  float kt;       // log2(e) / T
  float invT;     // 1 / T
  int kidcap;     // child slots per row record
  int rec_bytes;  // row record stride
  int wC;         // CTAs per sequence in the walk (its own vocabulary split)
  int wslice;     // vocabulary elements per walk CTA
};
// rows, sms, passA (bytes per logit that pass A reads): when given, rows
// that fill every SM and whose pass-A bytes fit L2 take one CTA each.
bool stream_geometry(int V, int tsz, int dsz, int* C, int* slice, int* nch, int* stages,
                     int64_t rows = 0, int sms = 0, int passA = 0);
cudaError_t launch_stream_bf16(StreamParams P, cudaStream_t st);
cudaError_t launch_stream_f32(StreamParams P, cudaStream_t st);

// Event pair around a dominant kernel launch (no-op unless profiling is on).
void prof_begin(int kind, cudaStream_t st);
void prof_end(int kind, cudaStream_t st);

cudaError_t launch_greedy(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st);
cudaError_t launch_sampled(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st);
// Single-launch chain verification for a few sequences (one cluster of 8
// CTAs per sequence, rows resident in shared memory): whether it applies,
// and its launch.
bool chain_small_fits(const VerifyShape& s, const VerifyArgs& a, int sms, int* slice,
                      size_t* smem);
cudaError_t launch_chain_small(const VerifyShape& s, const VerifyArgs& a, int slice, size_t smem,
                               cudaStream_t st);
// True when the call will be one single-cluster launch of that kernel, which
// then writes the status word itself (the caller skips clearing it).
bool chain_small_writes_status(const VerifyShape& s, const VerifyArgs& a);
bool sampled_supported(const VerifyShape& s, const VerifyArgs& a);
cudaError_t launch_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask,
                             uint64_t* bits, cudaStream_t st);
cudaError_t launch_philox(uint64_t seed, uint32_t offset, const int32_t* b, const int32_t* i,
                          const int32_t* slot, int n, float* out, cudaStream_t st);

// Target LM head: logits [M, V] (bf16, row stride ldo) = hidden [M, H] x
// W^T on tcgen05; with temperature > 0 and `stats`, also the per-row base-2
// log normalisers at that temperature into `lse` [M] (stats: [M, V/256]).
int lmhead_tiles_n(int V);
bool lmhead_supported(const void* hidden, const void* w, int H);
// test_stall: the producer withholds its first stage (bounded-wait test).
cudaError_t launch_lmhead(const void* hidden, const void* w, int M, int H, int V, float temperature,
                          uint16_t* logits, int64_t ldo, float2* stats, float* lse,
                          uint32_t* status, cudaStream_t st, bool test_stall = false);

// EAGLE-2 expand + rerank
struct Eagle2Cand {
  int32_t token;
  float logq;
};
cudaError_t launch_eagle2(const void* draft, int B, int V, int dtype, int depth, int topk,
                          int width, int total, float temperature, int32_t* node_tokens,
                          int32_t* parent, int32_t* q_row, float* value, uint8_t* mask,
                          float* draft_lse, Eagle2Cand* cand, uint32_t* status,
                          cudaStream_t st);

}  // namespace sv
