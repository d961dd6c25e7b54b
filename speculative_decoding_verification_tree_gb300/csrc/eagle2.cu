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

// One CTA per draft row: the row's `topk` most probable tokens and their
// log-probabilities log q = (z kt - log2 sum 2^(z kt)) ln 2 at temperature T
// (kt = log2(e) / T).  Aligned rows take one streaming pass in which every
// thread keeps its running maximum and the row's log-sum-exp; the k-th
// largest thread maximum is a lower bound on the k-th largest logit, so only
// the threads whose maximum reaches it rescan their own logits (recently
// read, from L2) and the candidates (every logit at or above the bound) are
// ranked exactly by (logit desc, index asc).  Rows where that leaves fewer
// than k or more than kCandCap candidates (ties, NaN, -inf) take the
// general streaming top-k shared with the top-k sampling path.
constexpr int kCandCap = 256;
constexpr int kFlagCap = 64;  // threads whose logits are rescanned
constexpr int kRowBatch = 4;  // 16-byte groups in flight per thread

template <typename T, bool kVec>
__global__ void __launch_bounds__(topk::kThreads) eagle2_rows(const T* __restrict__ x, int V,
                                                              int k, float kt,
                                                              Eagle2Cand* __restrict__ out,
                                                              uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ int32_t idx[SPEC_EAGLE2_MAX_TOPK];
  __shared__ float val[SPEC_EAGLE2_MAX_TOPK];
  __shared__ int cnt;
  __shared__ float lse;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_tau;
  __shared__ int s_nc, s_nf;
  __shared__ float red_m[topk::kWarps], red_z[topk::kWarps];
  const int64_t row = blockIdx.x;
  const T* rp = x + row * (int64_t)V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  topk::Cand* cbuf = reinterpret_cast<topk::Cand*>(smraw);
  bool fallback = !kVec;
  if constexpr (kVec) {
    constexpr int kU = sizeof(T) == 2 ? 1 : 2;  // uint4 per 8-logit group
    constexpr int kNT = topk::kThreads;
    const int G = V / 8;
    const uint4* base = reinterpret_cast<const uint4*>(rp);
    float mx = neg_inf();
    MaxSum ms{neg_inf(), 0.f};
    auto unpack = [&](const uint4 (&r)[kU], float (&v)[8]) {
      if constexpr (sizeof(T) == 2) {
        v[0] = bf16_lo(r[0].x); v[1] = bf16_hi(r[0].x); v[2] = bf16_lo(r[0].y); v[3] = bf16_hi(r[0].y);
        v[4] = bf16_lo(r[0].z); v[5] = bf16_hi(r[0].z); v[6] = bf16_lo(r[0].w); v[7] = bf16_hi(r[0].w);
      } else {
        v[0] = __uint_as_float(r[0].x); v[1] = __uint_as_float(r[0].y);
        v[2] = __uint_as_float(r[0].z); v[3] = __uint_as_float(r[0].w);
        v[4] = __uint_as_float(r[kU - 1].x); v[5] = __uint_as_float(r[kU - 1].y);
        v[6] = __uint_as_float(r[kU - 1].z); v[7] = __uint_as_float(r[kU - 1].w);
      }
    };
    for (int g0 = tid; g0 < G; g0 += kNT * kRowBatch) {
      uint4 r[kRowBatch][kU];
#pragma unroll
      for (int bI = 0; bI < kRowBatch; ++bI) {
        const int g = g0 + bI * kNT;
        if (g < G) {
#pragma unroll
          for (int u = 0; u < kU; ++u) r[bI][u] = topk::ldg_stream16(base + (int64_t)g * kU + u);
        }
      }
#pragma unroll
      for (int bI = 0; bI < kRowBatch; ++bI) {
        if (g0 + bI * kNT < G) {
          float v[8];
          unpack(r[bI], v);
          const float gm = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                                 fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
          mx = fmaxf(mx, gm);
          const float mt = __fmul_rn(gm, kt);
          if (mt > ms.m) {
            ms.z *= ex2(ms.m - mt);
            ms.m = mt;
          }
          if (ms.m != neg_inf()) {
            float z = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) z += ex2(fmaf(v[j], kt, -ms.m));
            ms.z += z;
          }
        }
      }
    }
    // log-sum-exp of the row
    ms = warp_ms(ms);
    if (lane == 0) {
      red_m[warp] = ms.m;
      red_z[warp] = ms.z;
    }
    // bound: k-th largest thread maximum (order keys; radix select by warp 0)
    const uint32_t mykey = topk::fkey(mx);
    cbuf[tid] = topk::Cand{mykey, tid};
    if (tid == 0) {
      s_nc = 0;
      s_nf = 0;
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t kth = 0u;
      topk::warp_select(cbuf, kNT, k, lane, hist, &kth);
      if (lane == 0) {
        s_tau = kth;
        MaxSum A{red_m[0], red_z[0]};
        for (int w = 1; w < topk::kWarps; ++w) A = ms_combine(A, MaxSum{red_m[w], red_z[w]});
        lse = A.m + log2f(A.z);
      }
    }
    __syncthreads();
    const uint32_t tau = s_tau;
    topk::Cand* cand = cbuf + kNT;  // after the bound's scratch
    int* flagged = reinterpret_cast<int*>(cand + kCandCap);
    if (mykey >= tau) {  // this thread holds a logit at or above the bound
      const int pos = atomicAdd(&s_nf, 1);
      if (pos < kFlagCap) flagged[pos] = tid;
    }
    __syncthreads();
    const int nf = s_nf;
    if (nf <= kFlagCap) {
      // the flagged threads' groups, rescanned by the whole CTA
      const int gpt = (G + kNT - 1) / kNT;
#pragma unroll 2
      for (int w = tid; w < nf * gpt; w += kNT) {
        const int f = w / gpt;
        const int g = flagged[f] + (w - f * gpt) * kNT;
        if (g < G) {
          uint4 r[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) r[u] = topk::ldg_stream16(base + (int64_t)g * kU + u);
          float v[8];
          unpack(r, v);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t kj = topk::fkey(v[j]);
            if (kj >= tau) {
              const int pos = atomicAdd(&s_nc, 1);
              if (pos < kCandCap) cand[pos] = topk::Cand{kj, g * 8 + j};
            }
          }
        }
      }
    }
    __syncthreads();
    const int nc = s_nc;
    fallback = (nf > kFlagCap || nc < k || nc > kCandCap || tau == 0u);
    if (!fallback) {
      // exact ranking of the candidates: logit desc, index asc
      for (int i = tid; i < nc; i += kNT) {
        const topk::Cand c = cand[i];
        int rk = 0;
        for (int j2 = 0; j2 < nc; ++j2) {
          const topk::Cand d = cand[j2];
          rk += topk::before(d.key, d.idx, c.key, c.idx) ? 1 : 0;
        }
        if (rk < k) {
          idx[rk] = c.idx;
          val[rk] = topk::funkey(c.key);
        }
      }
      if (tid == 0) cnt = k;
    }
    __syncthreads();
  }
  if (fallback) {
    topk::row_topk<T, kVec>(rp, V, k, kt, reinterpret_cast<topk::Cand*>(smraw), idx, val, &cnt,
                            &lse);
  }
  const int i = threadIdx.x;
  if (i < k) {
    Eagle2Cand* o = out + row * SPEC_EAGLE2_MAX_TOPK;
    o[i] = (i < cnt) ? Eagle2Cand{idx[i], fmaf(val[i], kt, -lse) * 0.69314718055994531f}
                     : Eagle2Cand{0, neg_inf()};
    if (i == 0 && (cnt < k || !(lse > neg_inf()) || isnan(lse)))
      flag_status(status, SPEC_STATUS_NAN);
  }
}

struct SelNode {
  float val;
  int tok, dep, id, par, row;
};

__device__ __forceinline__ bool sel_before(const SelNode& a, const SelNode& b) {
  if (a.val != b.val) return a.val > b.val;
  if (a.dep != b.dep) return a.dep < b.dep;
  return a.id < b.id;
}

__global__ void __launch_bounds__(kSelThreads) eagle2_select(const Eagle2Cand* __restrict__ cand,
                                                             int R, int depth, int topk, int width,
                                                             int total, int32_t* node_tokens,
                                                             int32_t* parent, int32_t* q_row,
                                                             float* value, uint32_t* status) {
  extern __shared__ unsigned char smraw[];
  SelNode* nd = reinterpret_cast<SelNode*>(smraw);
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
      int rk = 0;
      for (int j = 0; j < ln; ++j) rk += sel_before(nd[l0 + j], nd[l0 + i]) ? 1 : 0;
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
      nd[base + t] = SelNode{nd[pi].val + lq, e.token, d + 1, r * topk + c, pi, -1};
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
  for (int i = tid; i < n; i += blockDim.x) {
    int rk = 0;
    const SelNode me = nd[i];
    for (int j = 0; j < n; ++j) rk += sel_before(nd[j], me) ? 1 : 0;
    rank[i] = rk;
  }
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
                          Eagle2Cand* cand, uint32_t* status, cudaStream_t st) {
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
    kern<<<(unsigned)rows, topk::kThreads, rsm, st>>>(src, V, topk, kt, cand, status);
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
  const size_t smem = (size_t)kMaxCand * (sizeof(SelNode) + sizeof(int));
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
