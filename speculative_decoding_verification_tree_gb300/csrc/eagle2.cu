// EAGLE-2 dynamic draft tree: expand and rerank ("EAGLE-2: Faster Inference
// of Language Models with Dynamic Draft Trees", §4.1-4.2).
//
// value(node) = sum of log q along its root path (the product of draft
// confidences of §4.1, in the log domain).  Expand: each layer keeps its
// `width` best nodes; each kept node's draft row contributes its `topk` most
// probable tokens as children.  Rerank: all candidates by (value desc, depth
// asc, id asc), best `total` kept; a child never outranks its parent (its
// value is no larger and it is deeper), so the kept set is a connected tree
// and this order lists parents before children.
//
// Two kernels:
//  * eagle2_rows: one CTA per draft row, one HBM pass.  Log-sum-exp of z/T
//    (online, base 2) and the row's top-k tokens by logit, ties to the lower
//    index.  Each warp filters its contiguous part of the row against the
//    order key of its current k-th best and appends survivors to a shared
//    buffer, compacted when full; the CTA then merges the warps' lists.
//  * eagle2_select: one CTA per sequence.  Layer keeps and the rerank use
//    rank-by-counting over unique keys (deterministic), then write node
//    tokens, parents, q_row and values.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace sv {
namespace {

constexpr int kSelThreads = 512;
constexpr int kMaxCand = SPEC_EAGLE2_MAX_CANDIDATES;  // per sequence (host-checked)

// One CTA per draft row: the row's `topk` most probable tokens (bound-and-
// rescan streaming top-k shared with the top-k sampling path) and their
// log-probabilities log q = (z kt - log2 sum 2^(z kt)) ln 2 at temperature T
// (kt = log2(e) / T); the row's log2 normaliser goes to lse_out if given.
template <typename T, bool kVec>
__global__ void __launch_bounds__(topk::kThreads) eagle2_rows(const T* __restrict__ x, int V,
                                                              int k, float kt,
                                                              Eagle2Cand* __restrict__ out,
                                                              float* __restrict__ lse_out,
                                                              uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ int32_t idx[SPEC_EAGLE2_MAX_TOPK];
  __shared__ float val[SPEC_EAGLE2_MAX_TOPK];
  __shared__ int cnt;
  __shared__ float lse;
  const int64_t row = blockIdx.x;
  topk::row_topk_fast<T, kVec>(x + row * (int64_t)V, V, k, kt,
                               reinterpret_cast<topk::Cand*>(smraw), idx, val, &cnt, &lse,
                               0);  // long rows: the flagged threads' rescan
  const int i = threadIdx.x;
  if (i < k) {
    Eagle2Cand* o = out + row * SPEC_EAGLE2_MAX_TOPK;
    o[i] = (i < cnt) ? Eagle2Cand{idx[i], fmaf(val[i], kt, -lse) * 0.69314718055994531f}
                     : Eagle2Cand{0, neg_inf()};
    if (i == 0 && (cnt < k || !(lse > neg_inf()) || isnan(lse)))
      flag_status(status, SPEC_STATUS_NAN);
  }
  if (lse_out && i == 0) lse_out[row] = lse;
}

struct SelNode {
  float val;
  int tok, dep, id, par, row;
};

// Rank order of candidates: value descending, then depth, then candidate id
// ascending.  One 64-bit key per candidate whose ascending order is that
// order: the value's bits made monotone (-0 counts as +0; NaN values were
// made -inf), complemented, above depth (< 2^16) and id (< 2^16).
__device__ __forceinline__ uint64_t sel_key(float v, int dep, int id) {
  const uint32_t u = __float_as_uint(v + 0.f);
  const uint32_t up = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // grows with v
  return ((uint64_t)~up << 32) | ((uint64_t)(uint32_t)dep << 16) | (uint32_t)id;
}

// Number of keys in k[0, n) below `me` (4 independent counters).
__device__ __forceinline__ int count_below(const uint64_t* k, int n, uint64_t me) {
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0, j = 0;
  for (; j + 4 <= n; j += 4) {
    c0 += k[j] < me;
    c1 += k[j + 1] < me;
    c2 += k[j + 2] < me;
    c3 += k[j + 3] < me;
  }
  for (; j < n; ++j) c0 += k[j] < me;
  return (c0 + c1) + (c2 + c3);
}

__global__ void __launch_bounds__(kSelThreads) eagle2_select(const Eagle2Cand* __restrict__ cand,
                                                             int R, int depth, int topk, int width,
                                                             int total, int32_t* node_tokens,
                                                             int32_t* parent, int32_t* q_row,
                                                             float* value, uint32_t* status) {
  extern __shared__ unsigned char smraw[];
  uint64_t* key = reinterpret_cast<uint64_t*>(smraw);
  SelNode* nd = reinterpret_cast<SelNode*>(key + kMaxCand);
  int* rank = reinterpret_cast<int*>(nd + kMaxCand);
  __shared__ int kept[SPEC_EAGLE2_MAX_WIDTH];
  __shared__ int s_n, s_prev0, s_prevn;
  const int b = blockIdx.x, tid = threadIdx.x;
  const Eagle2Cand* cb = cand + (int64_t)b * R * SPEC_EAGLE2_MAX_TOPK;
  // layer 1: children of the root (draft row 0)
  for (int c = tid; c < topk; c += blockDim.x) {
    const Eagle2Cand e = cb[c];
    const float v = isnan(e.logq) ? neg_inf() : e.logq;
    nd[c] = SelNode{v, e.token, 1, c, -1, -1};
    key[c] = sel_key(v, 1, c);
  }
  if (tid == 0) {
    s_n = topk;
    s_prev0 = 0;
    s_prevn = topk;
  }
  __syncthreads();
  for (int d = 1; d <= depth; ++d) {
    const int l0 = s_prev0, ln = s_prevn;
    if (d == depth) break;
    // keep the `width` best of layer d (rank by counting within the layer)
    for (int i = tid; i < ln; i += blockDim.x) {
      const int rk = count_below(key + l0, ln, key[l0 + i]);
      if (rk < width) {
        kept[rk] = l0 + i;
        nd[l0 + i].row = 1 + (d - 1) * width + rk;
      }
    }
    __syncthreads();
    const int nk = min(width, ln);
    // layer d + 1: topk children of each kept node, from its draft row
    const int base = s_n;
    for (int t = tid; t < nk * topk; t += blockDim.x) {
      const int r = t / topk, c = t - r * topk;
      const int pi = kept[r];
      const int rw = nd[pi].row;
      const Eagle2Cand e = cb[(int64_t)rw * SPEC_EAGLE2_MAX_TOPK + c];
      const float lq = isnan(e.logq) ? neg_inf() : e.logq;
      const float v = nd[pi].val + lq;
      nd[base + t] = SelNode{v, e.token, d + 1, r * topk + c, pi, -1};
      key[base + t] = sel_key(v, d + 1, r * topk + c);
    }
    __syncthreads();
    if (tid == 0) {
      s_prev0 = base;
      s_prevn = nk * topk;
      s_n = base + nk * topk;
    }
    __syncthreads();
  }
  const int n = s_n;
  // rerank every candidate
  for (int i = tid; i < n; i += blockDim.x) rank[i] = count_below(key, n, key[i]);
  __syncthreads();
  if (tid == 0) q_row[(int64_t)b * (total + 1)] = 0;
  uint32_t bad = 0;
  for (int i = tid; i < n; i += blockDim.x) {
    const int j = rank[i];
    if (j >= total) continue;
    const SelNode me = nd[i];
    node_tokens[(int64_t)b * total + j] = me.tok;
    value[(int64_t)b * total + j] = me.val;
    int pj = -1;
    if (me.par >= 0) {
      pj = rank[me.par];
      if (pj >= j) bad |= SPEC_STATUS_BAD_TREE;  // cannot happen: parents rank first
    }
    parent[(int64_t)b * total + j] = pj;
    q_row[(int64_t)b * (total + 1) + j + 1] = me.row;
  }
  if (bad) flag_status(status, bad);
}

}  // namespace

cudaError_t launch_eagle2(const void* draft, int B, int V, int dtype, int depth, int topk,
                          int width, int total, float temperature, int32_t* node_tokens,
                          int32_t* parent, int32_t* q_row, float* value, uint8_t* mask,
                          float* draft_lse, Eagle2Cand* cand, uint32_t* status,
                          cudaStream_t st) {
  const int R = 1 + (depth - 1) * width;
  const float kt = kLog2e / temperature;
  const int64_t rows = (int64_t)B * R;
  const size_t esz = dtype == SPEC_BF16 ? 2 : 4;
  // vector path: whole groups of 8 elements, 16-byte aligned rows
  const bool vec = ((uintptr_t)draft % 16 == 0) && ((int64_t)V * esz % 16 == 0) && (V % 8 == 0);
  const size_t rsm = (size_t)topk::kWarps * topk::kBufCap * sizeof(topk::Cand);
  auto launch = [&](auto kern, const auto* src) -> cudaError_t {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm);
    if (err != cudaSuccess) return err;
    kern<<<(unsigned)rows, topk::kThreads, rsm, st>>>(src, V, topk, kt, cand, draft_lse, status);
    return cudaGetLastError();
  };
  prof_begin(SPEC_PROF_EXPAND, st);
  cudaError_t e;
  if (dtype == SPEC_BF16) {
    const uint16_t* src = (const uint16_t*)draft;
    e = vec ? launch(eagle2_rows<uint16_t, true>, src) : launch(eagle2_rows<uint16_t, false>, src);
  } else {
    const float* src = (const float*)draft;
    e = vec ? launch(eagle2_rows<float, true>, src) : launch(eagle2_rows<float, false>, src);
  }
  prof_end(SPEC_PROF_EXPAND, st);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)kMaxCand * (sizeof(uint64_t) + sizeof(SelNode) + sizeof(int));
  e = cudaFuncSetAttribute(eagle2_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  eagle2_select<<<B, kSelThreads, smem, st>>>(cand, R, depth, topk, width, total, node_tokens,
                                              parent, q_row, value, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (mask) return launch_tree_mask(parent, B, total, mask, nullptr, st);
  return cudaSuccess;
}

}  // namespace sv
