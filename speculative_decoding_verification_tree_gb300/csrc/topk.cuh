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
constexpr int kBufCap = 512;   // per-warp candidate buffer (entries)

// Order-preserving 32-bit key of a float (NaN -> 0, below every number).
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  if (isnan(v)) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float funkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint4 ldg_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct Cand {
  uint32_t key;
  int32_t idx;
};
__device__ __forceinline__ bool before(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Warp: keep the k best entries of buf[0, n) -- larger key first, equal keys
// by position -- in place and in their original order (buf is in increasing
// index order, so position order is index order).  The k-th best key is found
// by a 4-round radix select (8 bits per round, per-warp histogram `hist` of
// 256 counters), then one stable compaction pass keeps every key above it and
// the first `need` keys equal to it.  Returns min(n, k); *kth is the k-th best
// key (0 when n < k).
__device__ int warp_select(Cand* buf, int n, int k, int lane, uint32_t* hist, uint32_t* kth) {
  if (n < k) {
    *kth = 0u;
    return n;
  }
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t prefix = 0u;
  int need = k;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0u;
    __syncwarp();
    const uint32_t hmask = (shift == 24) ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int p = lane; p < n; p += 32) {
      const uint32_t key = buf[p].key;
      if ((key & hmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane l holds digits 255 - 8l down to 248 - 8l
    uint32_t c[8], lsum = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      lsum += c[j];
    }
    uint32_t incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - lsum;
    const bool mine = excl < (uint32_t)need && (uint32_t)need <= incl;
    uint32_t digit = 0u, above = 0u;
    if (mine) {
      uint32_t run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + c[j] >= (uint32_t)need) {
          digit = 255u - 8u * lane - j;
          above = run;
          break;
        }
        run += c[j];
      }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    digit = __shfl_sync(0xffffffffu, digit, src & 31);
    above = __shfl_sync(0xffffffffu, above, src & 31);
    prefix |= digit << shift;
    need -= (int)above;
    __syncwarp();
  }
  int out = 0, ties = 0;
  for (int base = 0; base < n; base += 32) {
    const int p = base + lane;
    const Cand c = (p < n) ? buf[p] : Cand{0u, -1};
    const bool gt = p < n && c.key > prefix;
    const bool eq = p < n && c.key == prefix;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const bool keep = gt || (eq && ties + __popc(eqm & lt) < need);
    const uint32_t km = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read its entry; writes go to lower slots
    if (keep) buf[out + __popc(km & lt)] = c;
    out += __popc(km);
    ties += __popc(eqm);
    __syncwarp();
  }
  *kth = prefix;
  return out;
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
  __shared__ uint32_t hist[kWarps][256];
  __shared__ float red_m[kWarps], red_z[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Cand* buf = smem + warp * kBufCap;
  const int groups = (V + 7) / 8;
  const int gpw = (groups + kWarps - 1) / kWarps;
  const int g0 = warp * gpw, g1 = min(groups, g0 + gpw);
  float thf = neg_inf();  // value of the warp's current k-th best
  int n = 0;
  MaxSum ms{neg_inf(), 0.f};
  // Rare path of a group: append its elements above the threshold (in index
  // order) and compact when the buffer is full.
  auto append = [&](int g, const float (&v)[8]) {
    int mine = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) mine += (g < g1 && g * 8 + j < V && v[j] > thf) ? 1 : 0;
    int pre = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += y;
    }
    const int tot = __shfl_sync(0xffffffffu, pre, 31);
    int pos = n + pre - mine;  // n <= kBufCap - 256 and tot <= 256: fits
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (g < g1 && g * 8 + j < V && v[j] > thf) buf[pos++] = Cand{fkey(v[j]), g * 8 + j};
    n += tot;
    __syncwarp();
    if (n > kBufCap - 256) {
      uint32_t kth;
      n = warp_select(buf, n, k, lane, hist[warp], &kth);
      if (n >= k) thf = funkey(kth);
    }
  };
  // Common path: log-sum-exp update and one ballot for the whole group.
  auto consume = [&](int g, const float (&v)[8]) {
    if (lse) {
      float mx = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                       fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
      const float mt = __fmul_rn(mx, kt);
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
    const bool c = (v[0] > thf) | (v[1] > thf) | (v[2] > thf) | (v[3] > thf) | (v[4] > thf) |
                   (v[5] > thf) | (v[6] > thf) | (v[7] > thf);
    if (__ballot_sync(0xffffffffu, c)) append(g, v);
  };
  if constexpr (kVec) {
    // aligned rows (V % 8 == 0): 16-byte loads three groups ahead
    constexpr int kU = sizeof(T) == 2 ? 1 : 2;  // uint4 per group
    const uint4* base = reinterpret_cast<const uint4*>(rp);
    uint4 r0[kU], r1[kU], r2[kU];
#define SV_TOPK_ISSUE(R, G)                                              \
    if ((G) < g1) {                                                      \
      _Pragma("unroll") for (int u = 0; u < kU; ++u)                      \
        R[u] = ldg_stream16(base + (int64_t)(G) * kU + u);               \
    }
#define SV_TOPK_STEP(R, S)                                               \
    if (gb + 32 * (S) < g1) {                                            \
      const int g = gb + 32 * (S) + lane;                                \
      float v[8];                                                        \
      if (g < g1) {                                                      \
        if constexpr (sizeof(T) == 2) {                                  \
          v[0] = bf16_lo(R[0].x); v[1] = bf16_hi(R[0].x);                \
          v[2] = bf16_lo(R[0].y); v[3] = bf16_hi(R[0].y);                \
          v[4] = bf16_lo(R[0].z); v[5] = bf16_hi(R[0].z);                \
          v[6] = bf16_lo(R[0].w); v[7] = bf16_hi(R[0].w);                \
        } else {                                                         \
          v[0] = __uint_as_float(R[0].x); v[1] = __uint_as_float(R[0].y);  \
          v[2] = __uint_as_float(R[0].z); v[3] = __uint_as_float(R[0].w);  \
          v[4] = __uint_as_float(R[kU - 1].x); v[5] = __uint_as_float(R[kU - 1].y); \
          v[6] = __uint_as_float(R[kU - 1].z); v[7] = __uint_as_float(R[kU - 1].w); \
        }                                                                \
      } else {                                                           \
        _Pragma("unroll") for (int j = 0; j < 8; ++j) v[j] = neg_inf();   \
      }                                                                  \
      SV_TOPK_ISSUE(R, g + 96)                                           \
      consume(g, v);                                                     \
    }
    SV_TOPK_ISSUE(r0, g0 + lane)
    SV_TOPK_ISSUE(r1, g0 + 32 + lane)
    SV_TOPK_ISSUE(r2, g0 + 64 + lane)
    for (int gb = g0; gb < g1; gb += 96) {
      SV_TOPK_STEP(r0, 0)
      SV_TOPK_STEP(r1, 1)
      SV_TOPK_STEP(r2, 2)
    }
#undef SV_TOPK_STEP
#undef SV_TOPK_ISSUE
  } else {
    for (int gb = g0; gb < g1; gb += 32) {
      const int g = gb + lane;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = (g < g1 && g * 8 + j < V) ? ElemIO<T>::get(rp, g * 8 + j) : neg_inf();
      consume(g, v);
    }
  }
  // Fewer than k elements above -inf in this warp's part (the threshold never
  // rose): the k best are completed by its -inf entries, lowest index first.
  if (n < k) {
    for (int gb = g0; gb < g1 && n < k; gb += 32) {
      const int g = gb + lane;
      int mine = 0;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = (g < g1 && g * 8 + j < V) ? ElemIO<T>::get(rp, g * 8 + j) : 0.f;
        mine += (g < g1 && g * 8 + j < V && v[j] == neg_inf()) ? 1 : 0;
      }
      int pre = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += y;
      }
      const int tot = __shfl_sync(0xffffffffu, pre, 31);
      int pos = n + pre - mine;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (g < g1 && g * 8 + j < V && v[j] == neg_inf()) {
          if (pos < kBufCap) buf[pos] = Cand{fkey(v[j]), g * 8 + j};
          ++pos;
        }
      n = min(n + tot, kBufCap);
      __syncwarp();
    }
  }
  {
    uint32_t unused;
    n = warp_select(buf, n, k, lane, hist[warp], &unused);
  }
  if (lse) ms = warp_ms(ms);
  if (lane == 0) {
    cnt[warp] = n;
    red_m[warp] = ms.m;
    red_z[warp] = ms.z;
  }
  __syncthreads();
  if (warp == 0) {
    // pack the lists to the front of the whole buffer area (moves are to
    // lower addresses; each 32-entry chunk is read before it is written)
    int m = cnt[0];
    for (int w = 1; w < kWarps; ++w) {
      const Cand* src = smem + w * kBufCap;
      for (int i0 = 0; i0 < cnt[w]; i0 += 32) {
        const int i = i0 + lane;
        Cand c{0u, -1};
        if (i < cnt[w]) c = src[i];
        __syncwarp();
        if (i < cnt[w]) smem[m + i] = c;
        __syncwarp();
      }
      m += cnt[w];
    }
    // the warps' lists concatenate in index order; select, then order the
    // kept entries best first (equal keys: lower index first)
    uint32_t unused;
    m = warp_select(buf, m, k, lane, hist[0], &unused);
    for (int i = lane; i < m; i += 32) {
      const Cand c = buf[i];
      int rk = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = buf[j].key;
        rk += (kj > c.key || (kj == c.key && j < i)) ? 1 : 0;
      }
      out_idx[rk] = c.idx;
      out_val[rk] = funkey(c.key);
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

// Bitonic sort of one 64-bit value per lane across the warp, descending:
// lane j ends with the (j + 1)-th largest.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      // in blocks that end up descending the lower lane keeps the larger
      const bool desc = (lane & size) == 0 || size == 32;
      const bool lower = (lane & stride) == 0;
      v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Streaming top-k, bound-and-rescan form (aligned rows).  One pass in which
// every thread keeps its running maximum (and, if lse is wanted, the row's
// log-sum-exp); the k-th largest thread maximum is a lower bound on the k-th
// largest logit, so only the threads whose maximum reaches it have logits at
// or above it: the CTA rescans just those threads' logits (recently read,
// from L2) and ranks the candidates exactly by (logit desc, index asc).
// Rows where that leaves fewer than k or more than kCandCap candidates (many
// ties at the bound, NaN, -inf) take row_topk.  Same outputs as row_topk.
constexpr int kCandCap = 1024;
constexpr int kRowBatch = 8;  // 16-byte groups in flight per thread
// Shared memory of row_topk_fast: the bound's sorted lists (2 KB), the
// flagged threads (1 KB), the candidates (kCandCap entries) and, from byte
// kGkOff, one 16-bit order key (top half of the key of its maximum) per
// 8-logit group, gk_slots groups per thread (0: rescan the flagged threads'
// groups instead); the fallback reuses it all.  gk_slots_for gives the slots
// an allocation holds.
constexpr size_t kGkOff = 4096 + kCandCap * sizeof(Cand);
constexpr int gk_slots_for(size_t smem_bytes) {
  return smem_bytes > kGkOff ? (int)((smem_bytes - kGkOff) / (kThreads * 2)) : 0;
}

// Nothing extra for the last warp to do (see row_topk_fast's `extra`).
struct NoExtra {
  __device__ void operator()(int) const {}
};

// `extra(lane)` runs once on the last warp, at the end, where that warp is
// usually idle (the ranking needs a thread per candidate).
template <typename T, bool kVec, int kBatch = kRowBatch, typename F = NoExtra>
__device__ void row_topk_fast(const T* __restrict__ rp, int V, int k, float kt, Cand* smem,
                              int32_t* out_idx, float* out_val, int* out_n, float* lse,
                              int gk_slots, F extra = F{}) {
  __shared__ uint32_t s_tau;
  __shared__ int s_nc, s_nf;
  __shared__ float red_m[kWarps], red_z[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  bool fallback = !kVec;
  if constexpr (kVec) {
    constexpr int kU = sizeof(T) == 2 ? 1 : 2;  // uint4 per 8-logit group
    constexpr int kNT = kThreads;
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
    // group maxima as 16-bit order keys, [slot][thread] (rows of at most
    // gk_slots groups per thread); the rescan then reloads only the groups
    // that can hold an entry at or above the bound
    uint16_t* gk = G <= gk_slots * kNT
                       ? reinterpret_cast<uint16_t*>(reinterpret_cast<unsigned char*>(smem) + kGkOff)
                       : nullptr;
    int slot0 = 0;
    for (int g0 = tid; g0 < G; g0 += kNT * kBatch, slot0 += kBatch) {
      uint4 r[kBatch][kU];
#pragma unroll
      for (int bI = 0; bI < kBatch; ++bI) {
        const int g = g0 + bI * kNT;
        if (g < G) {
#pragma unroll
          for (int u = 0; u < kU; ++u) r[bI][u] = ldg_stream16(base + (int64_t)g * kU + u);
        }
      }
#pragma unroll
      for (int bI = 0; bI < kBatch; ++bI) {
        if (g0 + bI * kNT < G) {
          float v[8];
          unpack(r[bI], v);
          const float gm = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                                 fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
          mx = fmaxf(mx, gm);
          if (gk) gk[(slot0 + bI) * kNT + tid] = (uint16_t)(fkey(gm) >> 16);
          if (lse) {
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
    }
    if (lse) {
      ms = warp_ms(ms);
      if (lane == 0) {
        red_m[warp] = ms.m;
        red_z[warp] = ms.z;
      }
    }
    // bound: the k-th largest thread maximum, exactly.  Each warp sorts its
    // 32 (key, thread) pairs (unique, thread ascending among equal keys);
    // every thread then counts the pairs above its own in the other warps'
    // sorted lists by binary search, and the thread of rank k - 1 holds the
    // bound.  No warp waits on another's serial selection.
    const uint32_t mykey = fkey(mx);
    uint64_t* lists = reinterpret_cast<uint64_t*>(smem);  // kNT entries
    {
      const uint64_t c = warp_sort_desc(((uint64_t)mykey << 32) | (uint32_t)(kNT - 1 - tid), lane);
      lists[warp * 32 + lane] = c;
      if (tid == 0) {
        s_nc = 0;
        s_nf = 0;
      }
      __syncthreads();
      int rank = lane;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        if (w2 == warp) continue;
        const uint64_t* L = lists + w2 * 32;
        int lo = 0;  // entries of L above c (L descending)
#pragma unroll
        for (int step = 16; step > 0; step >>= 1)
          if (L[lo + step - 1] > c) lo += step;
        rank += lo + ((lo == 31 && L[31] > c) ? 1 : 0);
      }
      if (rank == k - 1) s_tau = (uint32_t)(c >> 32);
      if (tid == 0 && lse) {
        MaxSum A{red_m[0], red_z[0]};
        for (int w = 1; w < kWarps; ++w) A = ms_combine(A, MaxSum{red_m[w], red_z[w]});
        *lse = A.m + log2f(A.z);
      }
    }
    __syncthreads();
    const uint32_t tau = s_tau;
    int* flagged = reinterpret_cast<int*>(smem + kNT);
    Cand* cand = smem + 2 * kNT;
    auto append_all = [&](int g, const float (&v)[8]) {  // one atomic per entry
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t kj = fkey(v[j]);
        if (kj >= tau) {
          const int pos = atomicAdd(&s_nc, 1);
          if (pos < kCandCap) cand[pos] = Cand{kj, g * 8 + j};
        }
      }
    };
    if (gk) {
      // each thread reloads its own groups whose key reaches the bound (the
      // group of its maximum, rarely more), two at most in registers with
      // one shared atomic per warp; more go through the per-entry path
      const uint32_t tau16 = tau >> 16;
      int nq = 0, ga = -1, gb = -1;
      if (mykey >= tau) {
        for (int j = 0, g = tid; g < G; ++j, g += kNT)
          if (gk[j * kNT + tid] >= tau16) {
            if (nq == 0) ga = g;
            else if (nq == 1) gb = g;
            ++nq;
          }
      }
      uint4 ra[kU], rb[kU];
      if (nq >= 1 && nq <= 2) {
#pragma unroll
        for (int u = 0; u < kU; ++u) ra[u] = ldg_stream16(base + (int64_t)ga * kU + u);
      }
      if (nq == 2) {
#pragma unroll
        for (int u = 0; u < kU; ++u) rb[u] = ldg_stream16(base + (int64_t)gb * kU + u);
      }
      float va[8], vb[8];
      int c = 0;
      if (nq >= 1 && nq <= 2) {
        unpack(ra, va);
#pragma unroll
        for (int j = 0; j < 8; ++j) c += fkey(va[j]) >= tau ? 1 : 0;
      }
      if (nq == 2) {
        unpack(rb, vb);
#pragma unroll
        for (int j = 0; j < 8; ++j) c += fkey(vb[j]) >= tau ? 1 : 0;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int wbase = 0;
      if (lane == 31 && incl > 0) wbase = atomicAdd(&s_nc, incl);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      int pos = wbase + incl - c;
      if (nq >= 1 && nq <= 2) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t kj = fkey(va[j]);
          if (kj >= tau) {
            if (pos < kCandCap) cand[pos] = Cand{kj, ga * 8 + j};
            ++pos;
          }
        }
      }
      if (nq == 2) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t kj = fkey(vb[j]);
          if (kj >= tau) {
            if (pos < kCandCap) cand[pos] = Cand{kj, gb * 8 + j};
            ++pos;
          }
        }
      }
      if (nq > 2) {
        for (int j = 0, g = tid; g < G; ++j, g += kNT)
          if (gk[j * kNT + tid] >= tau16) {
            uint4 r[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) r[u] = ldg_stream16(base + (int64_t)g * kU + u);
            float v[8];
            unpack(r, v);
            append_all(g, v);
          }
      }
    } else {
      if (mykey >= tau) flagged[atomicAdd(&s_nf, 1)] = tid;  // at most kNT entries
      __syncthreads();
      const int nf = s_nf;
      // the flagged threads' groups, rescanned by the whole CTA
      const int gpt = (G + kNT - 1) / kNT;
#pragma unroll 2
      for (int w = tid; w < nf * gpt; w += kNT) {
        const int f = w / gpt;
        const int g = flagged[f] + (w - f * gpt) * kNT;
        if (g < G) {
          uint4 r[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) r[u] = ldg_stream16(base + (int64_t)g * kU + u);
          float v[8];
          unpack(r, v);
          append_all(g, v);
        }
      }
    }
    __syncthreads();
    const int nc = s_nc;
    fallback = (nc < k || nc > kCandCap || tau == 0u);
    if (!fallback) {
      // exact ranking of the candidates: logit desc, index asc
      for (int i = tid; i < nc; i += kNT) {
        const Cand c = cand[i];
        int rk = 0;
#pragma unroll 8
        for (int j2 = 0; j2 < nc; ++j2) {
          const Cand d = cand[j2];
          rk += before(d.key, d.idx, c.key, c.idx) ? 1 : 0;
        }
        if (rk < k) {
          out_idx[rk] = c.idx;
          out_val[rk] = funkey(c.key);
        }
      }
      if (tid == 0) *out_n = k;
    }
    if (warp == kWarps - 1) extra(lane);
    __syncthreads();
  }
  if (fallback) row_topk<T, kVec>(rp, V, k, kt, smem, out_idx, out_val, out_n, lse);
  if constexpr (!kVec) {
    if (warp == kWarps - 1) extra(lane);
  }
}

}  // namespace
}  // namespace topk
}  // namespace sv
