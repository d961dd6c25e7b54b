// Chain verification of small batches in one launch.
//
// The method is the chain rule of "064 · 投机解码" (section 三) and of steps
// 3-4 in "投机解码与 EAGLE": p and q are the softmaxes of the transformed
// target and draft rows; drafted token x_k is accepted iff u_k < p_k(x_k) /
// q_k(x_k) (q = 0 accepts), left to right until the first rejection n; the
// emitted token is drawn by inverse CDF from norm(max(0, p_n - q_n)) (p_n when
// that has no mass) or, with no rejection, from p_K; alpha_k = sum min(p, q)
// is reported for every k.
//
// For a few sequences the streaming pipeline's three launches (records,
// streaming pass, walk) are mostly latency.  Here one cluster of 8 CTAs takes
// a whole sequence.  Each CTA copies its vocabulary slice of all K + 1 target
// and K draft rows into shared memory once (one bulk copy and one mbarrier
// per row, so work on a row starts as soon as it lands).  Row work is split
// into (row, part) items, one warp each, read as 4-element groups that a
// warp takes in 512-byte runs (no bank conflicts).  Two cluster barriers:
//   1. every row's (max, sum) partials, broadcast into every CTA;
//   2. alpha and the residual mass of every drafted row, p and q at the
//      drafted tokens and the status bits, broadcast into every CTA;
//   3. every CTA takes the same decisions from the same numbers (warp 0, a
//      lane per drafted token; rank 0 writes counts, masses and tokens) and
//      the same choice of the slice that holds the draw (from slice totals
//      it holds: residual masses, or sums of p from the row statistics);
//   4. that CTA finds the token: warp totals in order, then the warp's
//      4-element groups by a warp scan, then the element.
// Every wait is bounded and reports SPEC_STATUS_TIMEOUT.  A single-cluster
// launch (one sequence) writes the status word itself, so the caller need
// not clear it first.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kSC = 8;        // CTAs per sequence (vocabulary slices)
constexpr int kST = 512;      // threads per CTA
constexpr int kSW = kST / 32;
constexpr int kSMaxK = 16;    // drafted tokens per sequence served here
constexpr int kSRows = 2 * kSMaxK + 1;
constexpr size_t kSSmem = 200 * 1024;

enum { QS_LOGITS = 0, QS_PROBS_T1 = 1, QS_PROBS_T = 2 };

struct __align__(16) SmallSh {
  uint64_t bar[kSRows];        // one per copied row: target 0..K, then draft
  float2 part[kSRows][kSC];    // every CTA's (max, sum) per row
  float2 wpart[kSRows][kSW];   // this CTA's per-item partials [row][part]
  float2 xab[kSMaxK][kSC];     // every CTA's (alpha, residual mass)
  float2 xpq[kSMaxK];          // p and q at the drafted tokens
  uint32_t xbits[kSC];         // every CTA's status bits so far
  int tok[kSMaxK];             // the drafted tokens
  float uacc[kSMaxK], udraw[kSMaxK + 1];  // the decisions' uniforms
  float Lp[kSMaxK + 1], Lq[kSMaxK], invZq[kSMaxK];
  float wtot[kSW];
  int dec_sel, dec_n, dec_mode;  // the decision (the same in every CTA)
  float dec_t;
  uint32_t dec_bits;
  uint32_t cta_bits;
};

__device__ __forceinline__ void st_dsmem_f32x2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// address of this CTA's copy of a shared variable in the CTA of `rank`
__device__ __forceinline__ uint32_t at_rank(const void* p, uint32_t rank) {
  return mapa(smem_u32(p), rank);
}
// split cluster barrier: arrive early, wait where the peers must have started
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <typename T>
__device__ __forceinline__ float elem(const T* p, int i) {
  if constexpr (sizeof(T) == 2) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  else return reinterpret_cast<const float*>(p)[i];
}
// four consecutive elements from shared memory (element index a multiple of
// 4), or `fill` when they lie at or beyond `hi` (a multiple of 4)
template <typename T>
__device__ __forceinline__ void ld4s(const T* row, int e, int hi, float fill, float v[4]) {
  if (e >= hi) {
    v[0] = v[1] = v[2] = v[3] = fill;
    return;
  }
  if constexpr (sizeof(T) == 2) {
    const uint2 r = *reinterpret_cast<const uint2*>(row + e);
    v[0] = bf16_lo(r.x);
    v[1] = bf16_hi(r.x);
    v[2] = bf16_lo(r.y);
    v[3] = bf16_hi(r.y);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + e);
    v[0] = a.x;
    v[1] = a.y;
    v[2] = a.z;
    v[3] = a.w;
  }
}
// (max, sum 2^(v - max)) over elements lo..hi-1 of a row in shared memory,
// v = x kt (KIND 0: logits), the plain sum of x with max 0 (KIND 1:
// probabilities at T = 1) or v = log2(x) / T (KIND 2: probabilities); the
// warp's lanes take 4-element groups at lane * 4 and 128 + lane * 4 of every
// 256.  Returned in every lane.
template <typename T, int KIND>
__device__ __forceinline__ MaxSum part_stats(const T* row, int lo, int hi, int lane, float kt,
                                             float invT) {
  const float fill = KIND == 0 ? neg_inf() : 0.f;
  if (lo >= hi) return MaxSum{KIND == 1 ? 0.f : neg_inf(), 0.f};  // an empty part
  auto val = [&](float x) {
    return KIND == 0 ? __fmul_rn(x, kt) : (KIND == 1 ? x : __fmul_rn(lg2(x), invT));
  };
  if constexpr (KIND == 1) {
    float z0 = 0.f, z1 = 0.f;
    for (int e = lo + lane * 4; e < hi; e += 256) {
      float v[8];
      ld4s(row, e, hi, fill, v);
      ld4s(row, e + 128, hi, fill, v + 4);
      z0 += (v[0] + v[1]) + (v[2] + v[3]);
      z1 += (v[4] + v[5]) + (v[6] + v[7]);
    }
    return MaxSum{0.f, warp_sum(z0 + z1)};
  }
  // raw maxima start at the fill (log2(0) / T = -inf for probabilities)
  float m0 = fill, m1 = fill;
  for (int e = lo + lane * 4; e < hi; e += 256) {
    float v[8];
    ld4s(row, e, hi, fill, v);
    ld4s(row, e + 128, hi, fill, v + 4);
    m0 = fmaxf(m0, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
    m1 = fmaxf(m1, fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
  }
  // the max of the raw values gives the max of v (x kt and log2(x) / T are
  // increasing in x)
  const float M = val(warp_max(fmaxf(m0, m1)));
  if (M == neg_inf()) return MaxSum{neg_inf(), 0.f};
  float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
  for (int e = lo + lane * 4; e < hi; e += 256) {
    float v[8];
    ld4s(row, e, hi, fill, v);
    ld4s(row, e + 128, hi, fill, v + 4);
    z0 += ex2(val(v[0]) - M) + ex2(val(v[4]) - M);
    z1 += ex2(val(v[1]) - M) + ex2(val(v[5]) - M);
    z2 += ex2(val(v[2]) - M) + ex2(val(v[6]) - M);
    z3 += ex2(val(v[3]) - M) + ex2(val(v[7]) - M);
  }
  return MaxSum{M, warp_sum((z0 + z1) + (z2 + z3))};
}
// draft probability from the draft row's element y and its normaliser
template <int QK>
__device__ __forceinline__ float q_of(float y, float kt, float invT, float nLq, float iZ) {
  if constexpr (QK == QS_LOGITS) return ex2(fmaf(y, kt, nLq));
  else if constexpr (QK == QS_PROBS_T1) return __fmul_rn(y, iZ);
  else return ex2(fmaf(lg2(y), invT, nLq));
}
// value of a draft element that is not there (probability 0 after the transform)
template <int QK>
__device__ __forceinline__ float draft_fill() {
  return QK == QS_LOGITS ? neg_inf() : 0.f;
}

template <typename TT, typename TD, int QK>
__global__ void __launch_bounds__(kST, 1)
    chain_small(VerifyShape s, VerifyArgs a, int slice, float kt, float invT, int own_status) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ SmallSh sh;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / kSC;
  const int K = s.n, V = s.V, nrows = 2 * K + 1;
  const int r0 = (int)rank * slice;
  const int len = max(0, min(slice, V - r0));
  const TT* tsm = reinterpret_cast<const TT*>(dyn);
  const TD* dsm = reinterpret_cast<const TD*>(dyn + (size_t)(K + 1) * slice * sizeof(TT));
  uint32_t bits = 0;

  if (tid < nrows) {  // each initialising thread makes its barrier visible
    mbar_init(&sh.bar[tid], 1);
    fence_mbar_init();
  }
  if (tid == 0) sh.cta_bits = 0;
  cluster_arrive_relaxed();
  __syncthreads();
  if (tid == 0 && len > 0) {
    const uint32_t bt = (uint32_t)len * sizeof(TT), bd = (uint32_t)len * sizeof(TD);
    const TT* tg = reinterpret_cast<const TT*>(a.target);
    const TD* dg = reinterpret_cast<const TD*>(a.draft);
    for (int r = 0; r <= K; ++r) {
      mbar_expect_tx(&sh.bar[r], bt);
      bulk_g2s(const_cast<TT*>(tsm) + (size_t)r * slice,
               tg + ((int64_t)b * (K + 1) + r) * V + r0, bt, &sh.bar[r]);
    }
    for (int k = 0; k < K; ++k) {
      mbar_expect_tx(&sh.bar[K + 1 + k], bd);
      bulk_g2s(const_cast<TD*>(dsm) + (size_t)k * slice, dg + ((int64_t)b * K + k) * V + r0, bd,
               &sh.bar[K + 1 + k]);
    }
  }

  // the decisions' uniforms (Philox counters: sequence, position, slot),
  // by the last warp while the rows land
  if (w == kSW - 1 && lane <= K) {
    if (lane < K)
      sh.uacc[lane] = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b, (uint32_t)lane, 0);
    sh.udraw[lane] = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b, (uint32_t)lane, 1);
  }

  // 1. (max, sum) of every row: items (row, part), one warp each (about two
  //    per warp); a max pass, then a sum pass against that max, so no lane
  //    waits on a chain of rescales; per row the parts combined, then
  //    broadcast into every CTA of the cluster
  {
    const int P1 = min(kSW, (2 * kSW + nrows - 1) / nrows);
    const int plen = (len + P1 * 256 - 1) / (P1 * 256) * 256;
    for (int it = w; it < nrows * P1; it += kSW) {
      const int r = it / P1, pt = it % P1;
      const int lo = min(len, pt * plen), hi = min(len, lo + plen);
      if (len > 0 && !mbar_wait_bounded(&sh.bar[r], 0)) bits |= SPEC_STATUS_TIMEOUT;
      MaxSum A;
      if (r <= K) {
        A = part_stats<TT, 0>(tsm + (size_t)r * slice, lo, hi, lane, kt, invT);
      } else {
        A = part_stats<TD, QK == QS_LOGITS ? 0 : (QK == QS_PROBS_T1 ? 1 : 2)>(
            dsm + (size_t)(r - K - 1) * slice, lo, hi, lane, kt, invT);
      }
      if (lane == 0) sh.wpart[r][pt] = make_float2(A.m, A.z);
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started
    if (tid < nrows) {
      const bool plain = QK == QS_PROBS_T1 && tid > K;
      MaxSum A = plain ? MaxSum{0.f, 0.f} : MaxSum{neg_inf(), 0.f};
      const int P1 = min(kSW, (2 * kSW + nrows - 1) / nrows);
      for (int k = 0; k < P1; ++k) {
        const float2 v = sh.wpart[tid][k];
        if (plain) A.z += v.y;
        else A = ms_combine(A, MaxSum{v.x, v.y});
      }
      const uint32_t dst = smem_u32(&sh.part[tid][rank]);
#pragma unroll
      for (uint32_t c = 0; c < kSC; ++c) st_dsmem_f32x2(mapa(dst, c), make_float2(A.m, A.z));
    }
  }
  cluster_sync();
  if (tid < nrows) {
    const int r = tid;
    const bool plain = QK == QS_PROBS_T1 && r > K;
    MaxSum A = plain ? MaxSum{0.f, 0.f} : MaxSum{neg_inf(), 0.f};
#pragma unroll
    for (int c = 0; c < kSC; ++c) {
      const float2 v = sh.part[r][c];
      if (plain) A.z += v.y;
      else A = ms_combine(A, MaxSum{v.x, v.y});
    }
    if (!(A.z > 0.f) || isnan(A.z)) bits |= SPEC_STATUS_NAN;
    if (r <= K) {
      sh.Lp[r] = A.m + log2f(A.z);
    } else if (plain) {
      sh.invZq[r - K - 1] = 1.f / A.z;
      sh.Lq[r - K - 1] = 0.f;
    } else {
      sh.Lq[r - K - 1] = A.m + log2f(A.z);
      sh.invZq[r - K - 1] = 0.f;
    }
  }
  __syncthreads();

  // 2. acceptance mass and residual mass of every drafted row (items as in
  //    step 1); p and q at the drafted token from the CTA whose slice holds it
  {
    const int P2 = min(kSW, (2 * kSW + K - 1) / K);
    const int plen = (len + P2 * 256 - 1) / (P2 * 256) * 256;
    for (int it = w; it < K * P2; it += kSW) {
      const int k = it / P2, pt = it % P2;
      const int lo = min(len, pt * plen), hi = min(len, lo + plen);
      const TT* tr = tsm + (size_t)k * slice;
      const TD* dr = dsm + (size_t)k * slice;
      const float nLp = -sh.Lp[k], nLq = -sh.Lq[k], iZ = sh.invZq[k];
      float al[4] = {0.f, 0.f, 0.f, 0.f}, rl[4] = {0.f, 0.f, 0.f, 0.f};
      for (int e = lo + lane * 4; e < hi; e += 256) {
        float x[8], y[8];
        ld4s(tr, e, hi, neg_inf(), x);
        ld4s(tr, e + 128, hi, neg_inf(), x + 4);
        ld4s(dr, e, hi, draft_fill<QK>(), y);
        ld4s(dr, e + 128, hi, draft_fill<QK>(), y + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p = ex2(fmaf(x[i], kt, nLp));
          const float mn = fminf(p, q_of<QK>(y[i], kt, invT, nLq, iZ));
          al[i & 3] += mn;
          rl[i & 3] += p - mn;
        }
      }
      const float als = warp_sum((al[0] + al[1]) + (al[2] + al[3]));
      const float rls = warp_sum((rl[0] + rl[1]) + (rl[2] + rl[3]));
      if (lane == 0) sh.wpart[k][pt] = make_float2(als, rls);
    }
    __syncthreads();
    if (tid < K) {
      const int k = tid;
      float A = 0.f, Rm = 0.f;
      for (int c = 0; c < P2; ++c) {
        A += sh.wpart[k][c].x;
        Rm += sh.wpart[k][c].y;
      }
      const uint32_t dab = smem_u32(&sh.xab[k][rank]);
#pragma unroll
      for (uint32_t c = 0; c < kSC; ++c) st_dsmem_f32x2(mapa(dab, c), make_float2(A, Rm));
      const int x = a.node_tokens[(int64_t)b * K + k];
      sh.tok[k] = x;
      if (x >= r0 && x < r0 + len) {
        const float px = ex2(fmaf(elem(tsm + (size_t)k * slice, x - r0), kt, -sh.Lp[k]));
        const float qx = q_of<QK>(elem(dsm + (size_t)k * slice, x - r0), kt, invT, -sh.Lq[k],
                                  sh.invZq[k]);
        const uint32_t dpq = smem_u32(&sh.xpq[k]);
#pragma unroll
        for (uint32_t c = 0; c < kSC; ++c) st_dsmem_f32x2(mapa(dpq, c), make_float2(px, qx));
      }
    }
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits) atomicOr(&sh.cta_bits, bits);
  __syncthreads();
  if (tid < kSC) st_dsmem_u32(at_rank(&sh.xbits[rank], (uint32_t)tid), sh.cta_bits);
  cluster_sync();  // the last cluster barrier: no peer touches this CTA after it

  // 3. decisions, outputs and the slice of the draw: warp 0 of every CTA
  //    from the same numbers (lane k tests drafted token k, lane c < 8 holds
  //    slice c's draw mass); rank 0 writes the outputs
  if (w == 0) {
    uint32_t all = __reduce_or_sync(0xffffffffu, lane < kSC ? sh.xbits[lane] : 0u);
    uint32_t fl = 0;
    bool rej = false;
    float A = 0.f;
    if (lane < K) {
#pragma unroll
      for (int c = 0; c < kSC; ++c) A += sh.xab[lane][c].x;
      const int x = sh.tok[lane];
      bool acc;
      if (x < 0 || x >= V) {
        fl |= SPEC_STATUS_TOKEN_RANGE;
        acc = false;
      } else {
        const float px = sh.xpq[lane].x, qx = sh.xpq[lane].y;
        if (qx == 0.f) {
          fl |= SPEC_STATUS_QZERO_ACCEPT;
          acc = true;
        } else {
          acc = sh.uacc[lane] < px / qx;
        }
        // a rejected token leaves the draft without its mass: none left
        if (!acc && !(1.f - qx > 0.f)) fl |= SPEC_STATUS_DRAFT_EXHAUSTED;
      }
      rej = !acc;
    }
    const uint32_t rb = __ballot_sync(0xffffffffu, rej);
    const int n = rb ? __ffs(rb) - 1 : K;
    all |= __reduce_or_sync(0xffffffffu, lane <= n ? fl : 0u);  // the chain stops at n
    // the draw's weights: residual of row n, else p of row n (no residual
    // mass, flagged) or of row K (every draft accepted)
    const float Rm = warp_sum((n < K && lane < kSC) ? sh.xab[n][lane].y : 0.f);
    const int mode = (n < K && Rm > 0.f) ? 0 : 1;
    if (n < K && !(Rm > 0.f)) all |= SPEC_STATUS_RESIDUAL_ZERO;
    float wc = 0.f;
    if (lane < kSC) {
      if (mode == 0) {
        wc = sh.xab[n][lane].y;
      } else {
        const float2 v = sh.part[n][lane];
        wc = v.x == neg_inf() ? 0.f : v.y * ex2(v.x - sh.Lp[n]);
      }
    }
    float inc = wc;  // inclusive scan over the slices, in order
#pragma unroll
    for (int o = 1; o < kSC; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const float tot = __shfl_sync(0xffffffffu, inc, kSC - 1);
    const float t = sh.udraw[n] * tot;
    const bool pos = lane < kSC && wc > 0.f;
    const uint32_t hit = __ballot_sync(0xffffffffu, pos && inc > t);
    const uint32_t posb = __ballot_sync(0xffffffffu, pos);
    const float before = inc - wc;  // mass of the slices below this one
    int sel = -1;
    float tl = 0.f;
    if (hit) {
      sel = __ffs(hit) - 1;
      tl = t - __shfl_sync(0xffffffffu, before, sel);
    } else if (posb) {  // rounding: the last slice with mass, its last token
      sel = 31 - __clz(posb);
      tl = 3.0e38f;
      all |= SPEC_STATUS_CDF_FALLBACK;
    }
    if (rank == 0) {
      if (lane < K) a.mass[(int64_t)b * K + lane] = A;
      if (lane == 0) a.count[b] = n;
      int32_t* out = a.out_tokens + (int64_t)b * (K + 1);
      if (lane <= K) {
        if (lane < n) out[lane] = sh.tok[lane];
        else if (lane > n) out[lane] = -1;
        else if (sel < 0) out[lane] = 0;  // no mass anywhere (NaN rows, flagged)
      }
    }
    if (lane == 0) {
      sh.dec_sel = sel;
      sh.dec_n = n;
      sh.dec_mode = mode;
      sh.dec_t = tl;
      sh.dec_bits = all;
    }
  }
  __syncthreads();
  // the CTA that holds the draw finishes the call (rank 0 when nothing has mass)
  if ((sh.dec_sel < 0 ? 0 : sh.dec_sel) != (int)rank) return;

  // 4. inverse CDF inside the owning slice, in vocabulary order: warp parts
  //    in order, then the warp's 4-element groups (a warp scan per run of
  //    128 logits), then the group's elements
  const int n = sh.dec_n, mode = sh.dec_mode;
  if (tid == 0) sh.cta_bits = 0;
  if (sh.dec_sel >= 0) {
    const TT* tr = tsm + (size_t)n * slice;
    const TD* dr = dsm + (size_t)(n < K ? n : 0) * slice;
    const float nLp = -sh.Lp[n];
    const float nLq = n < K ? -sh.Lq[n] : 0.f, iZ = n < K ? sh.invZq[n] : 0.f;
    // weights of the group at e (zero beyond hi)
    auto group = [&](int e, int hi, float wv[4]) {
      float x[4];
      ld4s(tr, e, hi, neg_inf(), x);
      if (mode == 0) {
        float y[4];
        ld4s(dr, e, hi, draft_fill<QK>(), y);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          wv[i] = fmaxf(0.f, ex2(fmaf(x[i], kt, nLp)) - q_of<QK>(y[i], kt, invT, nLq, iZ));
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) wv[i] = ex2(fmaf(x[i], kt, nLp));
      }
    };
    const int dsub = (len + kSW * 128 - 1) / (kSW * 128) * 128;
    const int lo = min(len, w * dsub), hi = min(len, lo + dsub);
    float mine = 0.f;
    for (int e = lo + lane * 4; e < hi; e += 128) {
      float wv[4];
      group(e, hi, wv);
      mine += (wv[0] + wv[1]) + (wv[2] + wv[3]);
    }
    mine = warp_sum(mine);
    if (lane == 0) sh.wtot[w] = mine;
    __syncthreads();
    // the warp whose part passes the threshold (every thread finds the same)
    const float tl = sh.dec_t;
    float run = 0.f;
    int sw = -1, lastw = -1;
    for (int k = 0; k < kSW; ++k) {
      const float v = sh.wtot[k];
      if (v > 0.f) {
        lastw = k;
        if (sw < 0 && run + v > tl) sw = k;
      }
      if (sw < 0) run += v;
    }
    bool fallback = false;
    if (sw < 0) {  // rounding: the last part with mass, its last positive token
      sw = lastw;
      fallback = true;
    }
    if (w == sw) {
      const float tt = fallback ? 3.0e38f : tl;
      int pick = -1, lastp = -1;
      for (int e0 = lo; e0 < hi && pick < 0; e0 += 128) {
        const int e = e0 + lane * 4;
        float wv[4];
        group(e, hi, wv);
        const float gs = (wv[0] + wv[1]) + (wv[2] + wv[3]);
        float inc = gs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const uint32_t hitl = __ballot_sync(0xffffffffu, gs > 0.f && run + inc > tt);
        const uint32_t posl = __ballot_sync(0xffffffffu, gs > 0.f);
        if (hitl) {
          const int l = __ffs(hitl) - 1;
          if (lane == l) {  // the element within the group
            float c = run + inc - gs;
            int lp = -1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              c += wv[i];
              if (wv[i] > 0.f) {
                lp = e + i;
                if (pick < 0 && c > tt) pick = e + i;
              }
            }
            if (pick < 0) {  // rounding inside the group
              pick = lp;
              atomicOr(&sh.cta_bits, SPEC_STATUS_CDF_FALLBACK);
            }
          }
          pick = __shfl_sync(0xffffffffu, pick, l);
        } else if (posl) {
          const int l = 31 - __clz(posl);  // last group with mass so far
          int lp = -1;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (wv[i] > 0.f) lp = e + i;
          lastp = __shfl_sync(0xffffffffu, lp, l);
        }
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) {
        if (pick < 0) {
          pick = lastp;
          atomicOr(&sh.cta_bits, SPEC_STATUS_CDF_FALLBACK);
        }
        a.out_tokens[(int64_t)b * (K + 1) + n] = r0 + (pick < 0 ? 0 : pick);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t all = sh.dec_bits | sh.cta_bits;
    if (own_status) *a.status = all;  // the only cluster: the whole word
    else if (all) atomicOr(a.status, all);
  }
}

template <typename TT, typename TD>
cudaError_t launch_t(const VerifyShape& s, const VerifyArgs& a, int slice, size_t smem,
                     cudaStream_t st) {
  const float T = a.prm.temperature;
  const int qk = a.prm.draft_kind == SPEC_DRAFT_LOGITS ? QS_LOGITS
                                                       : (T == 1.f ? QS_PROBS_T1 : QS_PROBS_T);
  auto kern = qk == QS_LOGITS ? chain_small<TT, TD, QS_LOGITS>
                              : (qk == QS_PROBS_T1 ? chain_small<TT, TD, QS_PROBS_T1>
                                                   : chain_small<TT, TD, QS_PROBS_T>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(s.B * kSC));
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(SPEC_PROF_VERIFY, st);
  e = cudaLaunchKernelEx(&cfg, kern, s, a, slice, kLog2e / T, 1.f / T, s.B == 1 ? 1 : 0);
  prof_end(SPEC_PROF_VERIFY, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// The single-launch path applies: a sampled chain without truncation, 1 to
// kSMaxK drafts, 16-byte aligned rows with V a multiple of 8, one wave of
// clusters, and every row's slice resident in shared memory.
bool chain_small_fits(const VerifyShape& s, const VerifyArgs& a, int sms, int* slice, size_t* smem) {
  if (!s.chain || s.B < 1 || s.n < 1 || s.n > kSMaxK) return false;
  if (!(a.prm.temperature > 0.f) || truncation_k(&a.prm, s.V) > 0 || !a.draft || a.tlse)
    return false;
  if ((int64_t)s.B * kSC > sms) return false;
  const int tsz = a.dt_target == SPEC_BF16 ? 2 : 4, dsz = a.dt_draft == SPEC_BF16 ? 2 : 4;
  if (s.V % 8 != 0 || (uintptr_t)a.target % 16 != 0 || (uintptr_t)a.draft % 16 != 0) return false;
  const int sl = ((s.V + kSC - 1) / kSC + 7) / 8 * 8;
  const size_t need = (size_t)(s.n + 1) * sl * tsz + (size_t)s.n * sl * dsz;
  if (need > kSSmem) return false;
  *slice = sl;
  *smem = need;
  return true;
}

bool chain_small_writes_status(const VerifyShape& s, const VerifyArgs& a) {
  if (s.B != 1) return false;
  int dev = 0, sms = 0, sl = 0;
  size_t sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return chain_small_fits(s, a, sms, &sl, &sm);
}

cudaError_t launch_chain_small(const VerifyShape& s, const VerifyArgs& a, int slice, size_t smem,
                               cudaStream_t st) {
  if (a.dt_target == SPEC_BF16) {
    if (a.dt_draft == SPEC_BF16) return launch_t<uint16_t, uint16_t>(s, a, slice, smem, st);
    return launch_t<uint16_t, float>(s, a, slice, smem, st);
  }
  if (a.dt_draft == SPEC_BF16) return launch_t<float, uint16_t>(s, a, slice, smem, st);
  return launch_t<float, float>(s, a, slice, smem, st);
}

}  // namespace sv
