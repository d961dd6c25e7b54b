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

namespace sv {
namespace {

constexpr int kRowsThreads = 256;
constexpr int kRowsWarps = kRowsThreads / 32;
constexpr int kBufCap = 512;   // per-warp candidate buffer
constexpr int kSelThreads = 512;
constexpr int kMaxCand = SPEC_EAGLE2_MAX_CANDIDATES;  // per sequence (host-checked)

// Order-preserving 32-bit key of a float (NaN -> 0, below every number).
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  if (isnan(v)) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct Cand {
  uint32_t key;
  int32_t idx;
};
// (ka, ia) ranks before (kb, ib): larger key, then lower index.
__device__ __forceinline__ bool before(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Warp: keep the k best entries of buf[0, n) in buf[0, k) (sorted); returns
// the new count (min(n, k)).  All lanes participate.
__device__ int warp_compact(Cand* buf, int n, int k, int lane) {
  const int m = min(n, k);
  // k rounds of warp-wide selection; picked entries are marked by idx = -1
  Cand out_l = {0u, INT_MAX};
  for (int r = 0; r < m; ++r) {
    uint32_t bk = 0u;
    int bi = INT_MAX, bp = -1;
    for (int p = lane; p < n; p += 32) {
      const Cand c = buf[p];
      if (c.idx >= 0 && (bp < 0 || before(c.key, c.idx, bk, bi))) {
        bk = c.key;
        bi = c.idx;
        bp = p;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int op = __shfl_xor_sync(0xffffffffu, bp, o);
      if (op >= 0 && (bp < 0 || before(ok, oi, bk, bi))) {
        bk = ok;
        bi = oi;
        bp = op;
      }
    }
    if (lane == r % 32 && r < 32) out_l = Cand{bk, bi};
    if (lane == 0 && bp >= 0) buf[bp].idx = -1;
    __syncwarp();
  }
  if (lane < m) buf[lane] = out_l;
  __syncwarp();
  return m;
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(kRowsThreads) eagle2_rows(const T* __restrict__ x, int V,
                                                            int topk, float kt,
                                                            Eagle2Cand* __restrict__ out,
                                                            uint32_t* status) {
  __shared__ Cand buf[kRowsWarps][kBufCap];
  __shared__ int cnt[kRowsWarps];
  __shared__ float red_m[kRowsWarps], red_z[kRowsWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const T* rp = x + row * (int64_t)V;
  // contiguous part of the row per warp, in groups of 8 elements per lane
  const int groups = (V + 7) / 8;
  const int gpw = (groups + kRowsWarps - 1) / kRowsWarps;
  const int g0 = warp * gpw, g1 = min(groups, g0 + gpw);
  if (lane == 0) cnt[warp] = 0;
  __syncwarp();
  uint32_t th = 0u;  // order key of the warp's current k-th best (0: none)
  int n = 0;
  MaxSum ms{neg_inf(), 0.f};
  for (int gb = g0; gb < g1; gb += 32) {
    const int g = gb + lane;
    float v[8];
    if (g < g1) {
      const int e = g * 8;
      if constexpr (kVec) {
        if constexpr (sizeof(T) == 2) {
          const uint4 w = *reinterpret_cast<const uint4*>(rp + e);
          v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
          v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
        } else {
          const float4 a = *reinterpret_cast<const float4*>(rp + e);
          const float4 b = *reinterpret_cast<const float4*>(rp + e + 4);
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
          v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (e + j < V) ? ElemIO<T>::get(rp, e + j) : neg_inf();
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = neg_inf();
    }
    // log-sum-exp (base 2)
    float mt = neg_inf();
#pragma unroll
    for (int j = 0; j < 8; ++j) mt = fmaxf(mt, __fmul_rn(v[j], kt));
    if (mt > ms.m) {
      ms.z *= ex2(ms.m - mt);
      ms.m = mt;
    }
    if (ms.m != neg_inf()) {
#pragma unroll
      for (int j = 0; j < 8; ++j) ms.z += ex2(fmaf(v[j], kt, -ms.m));
    }
    // candidates above the warp threshold (elements past V are -inf, whose
    // key is above NaN's; they are excluded by index)
    int mine = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mine += (g < g1 && g * 8 + j < V && fkey(v[j]) > th) ? 1 : 0;
    if (__ballot_sync(0xffffffffu, mine)) {
      int pre = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += y;
      }
      const int tot = __shfl_sync(0xffffffffu, pre, 31);
      if (n + tot > kBufCap) {  // cannot happen: compaction keeps n <= kBufCap - 256
        n = kBufCap - tot;
      }
      int pos = n + pre - mine;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (g < g1 && g * 8 + j < V && fkey(v[j]) > th) buf[warp][pos++] = Cand{fkey(v[j]), g * 8 + j};
      }
      n += tot;
      __syncwarp();
      if (n > kBufCap - 256) {
        n = warp_compact(buf[warp], n, topk, lane);
        th = (n >= topk) ? buf[warp][topk - 1].key : 0u;
      }
    }
  }
  n = warp_compact(buf[warp], n, topk, lane);
  ms = warp_ms(ms);
  if (lane == 0) {
    cnt[warp] = n;
    red_m[warp] = ms.m;
    red_z[warp] = ms.z;
  }
  __syncthreads();
  if (warp == 0) {
    // merge the warps' lists into warp 0's buffer, then select
    int m = cnt[0];
    for (int w = 1; w < kRowsWarps; ++w) {
      for (int i = lane; i < cnt[w]; i += 32) buf[0][m + i] = buf[w][i];
      m += cnt[w];
    }
    __syncwarp();
    m = warp_compact(buf[0], m, topk, lane);
    MaxSum A{red_m[0], red_z[0]};
    for (int w = 1; w < kRowsWarps; ++w) A = ms_combine(A, MaxSum{red_m[w], red_z[w]});
    const float L2 = A.m + log2f(A.z);  // log2 sum 2^(z kt)
    const bool bad = !(A.z > 0.f) || isnan(A.z) || m < topk;
    if (lane == 0 && bad) flag_status(status, SPEC_STATUS_NAN);
    Eagle2Cand* o = out + row * SPEC_EAGLE2_MAX_TOPK;
    for (int i = lane; i < topk; i += 32) {
      if (i < m) {
        const int idx = buf[0][i].idx;
        const float z = ElemIO<T>::get(rp, idx);
        // natural-log probability: (z kt - L2) * ln 2
        o[i] = Eagle2Cand{idx, (fmaf(z, kt, -L2)) * 0.69314718055994531f};
      } else {
        o[i] = Eagle2Cand{0, neg_inf()};
      }
    }
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
  prof_begin(SPEC_PROF_EXPAND, st);
  if (dtype == SPEC_BF16) {
    if (vec)
      eagle2_rows<uint16_t, true><<<(unsigned)rows, kRowsThreads, 0, st>>>(
          (const uint16_t*)draft, V, topk, kt, cand, status);
    else
      eagle2_rows<uint16_t, false><<<(unsigned)rows, kRowsThreads, 0, st>>>(
          (const uint16_t*)draft, V, topk, kt, cand, status);
  } else {
    if (vec)
      eagle2_rows<float, true><<<(unsigned)rows, kRowsThreads, 0, st>>>(
          (const float*)draft, V, topk, kt, cand, status);
    else
      eagle2_rows<float, false><<<(unsigned)rows, kRowsThreads, 0, st>>>(
          (const float*)draft, V, topk, kt, cand, status);
  }
  cudaError_t e = cudaGetLastError();
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
