// Streaming top-k of one logit row per CTA (k <= 128), ties to the lower
// index -- the "keep the k largest logits" step of the sampling transform
// ("064 · 投机解码", section 二: p and q include the top-k / nucleus
// transform).
//
// One HBM pass.  Each warp owns a contiguous part of the row and keeps the
// order keys of its candidates in a shared buffer: an element enters only if
// its key beats the warp's current k-th best (so after the first few hundred
// elements almost nothing enters), and the buffer is compacted to its k best
// when it fills.  The CTA then merges the warps' lists.  Elements are visited
// in increasing index order within a warp, so a later element equal to the
// current k-th best can never belong to the top k: the strict comparison is
// exact, ties included.
#pragma once

#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace topk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 128;
constexpr int kBufCap = 1024;  // per-warp candidate buffer (entries)

// Order-preserving 32-bit key of a float (NaN -> 0, below every number).
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  if (isnan(v)) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float funkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct Cand {
  uint32_t key;
  int32_t idx;
};
__device__ __forceinline__ bool before(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Warp: keep the k best entries of buf[0, n) in buf[0, min(n, k)), sorted.
__device__ int warp_compact(Cand* buf, int n, int k, int lane) {
  const int m = min(n, k);
  Cand keep[kMaxK / 32];
#pragma unroll
  for (int i = 0; i < kMaxK / 32; ++i) keep[i] = Cand{0u, INT_MAX};
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
#pragma unroll
    for (int i = 0; i < kMaxK / 32; ++i)
      if (r == i * 32 + lane) keep[i] = Cand{bk, bi};
    if (lane == 0 && bp >= 0) buf[bp].idx = -1;
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < kMaxK / 32; ++i)
    if (i * 32 + lane < m) buf[i * 32 + lane] = keep[i];
  __syncwarp();
  return m;
}

// Top-k of the row at `rp` (V logits); smem holds kWarps * kBufCap Cands.
// Writes the k best (index, logit) pairs, best first, to out_idx / out_val
// (count in *out_n; fewer than k only when the row has fewer non-NaN
// entries).  If lse != nullptr also returns log2(sum 2^(z kt)) of the row.
// All threads of the CTA must call.
template <typename T, bool kVec>
__device__ void row_topk(const T* __restrict__ rp, int V, int k, float kt, Cand* smem,
                         int32_t* out_idx, float* out_val, int* out_n, float* lse) {
  __shared__ int cnt[kWarps];
  __shared__ float red_m[kWarps], red_z[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Cand* buf = smem + warp * kBufCap;
  const int groups = (V + 7) / 8;
  const int gpw = (groups + kWarps - 1) / kWarps;
  const int g0 = warp * gpw, g1 = min(groups, g0 + gpw);
  uint32_t th = 0u;  // key of the warp's current k-th best (0: none yet)
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
    if (lse) {
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
    }
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
      int pos = n + pre - mine;  // n <= kBufCap - 256 and tot <= 256: fits
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (g < g1 && g * 8 + j < V && fkey(v[j]) > th) buf[pos++] = Cand{fkey(v[j]), g * 8 + j};
      }
      n += tot;
      __syncwarp();
      if (n > kBufCap - 256) {
        n = warp_compact(buf, n, k, lane);
        th = (n >= k) ? buf[k - 1].key : 0u;
      }
    }
  }
  n = warp_compact(buf, n, k, lane);
  if (lse) ms = warp_ms(ms);
  if (lane == 0) {
    cnt[warp] = n;
    red_m[warp] = ms.m;
    red_z[warp] = ms.z;
  }
  __syncthreads();
  if (warp == 0) {
    int m = cnt[0];
    for (int w = 1; w < kWarps; ++w) {
      for (int i = lane; i < cnt[w]; i += 32) buf[m + i] = smem[w * kBufCap + i];
      m += cnt[w];
    }
    __syncwarp();
    m = warp_compact(buf, m, k, lane);
    for (int i = lane; i < m; i += 32) {
      out_idx[i] = buf[i].idx;
      out_val[i] = funkey(buf[i].key);
    }
    if (lane == 0) {
      *out_n = m;
      if (lse) {
        MaxSum A{red_m[0], red_z[0]};
        for (int w = 1; w < kWarps; ++w) A = ms_combine(A, MaxSum{red_m[w], red_z[w]});
        *lse = A.m + log2f(A.z);
      }
    }
  }
  __syncthreads();
}

}  // namespace
}  // namespace topk
}  // namespace sv
