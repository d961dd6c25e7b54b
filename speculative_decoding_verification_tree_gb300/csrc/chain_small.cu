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
// and K draft rows into shared memory once (bulk copies on one mbarrier);
// each of its warps owns one eighth of the slice in every row, so the row
// reductions need no block barrier.  Then, one cluster barrier each:
//   1. every row's (max, sum) partials, broadcast into every CTA;
//   2. alpha and the residual mass of every drafted row, and p and q at the
//      drafted tokens, into rank 0;
//   3. rank 0 decides, writes counts, masses and accepted tokens, and picks
//      the CTA whose slice holds the draw (from slice totals it already
//      holds: residual masses, or sums of p from the row statistics);
//   4. that CTA finds the token in its slice (per-thread ranges in order).
// Every wait is bounded and reports SPEC_STATUS_TIMEOUT.  A single-cluster
// launch (one sequence) writes the status word itself, so the caller need
// not clear it first.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kSC = 8;        // CTAs per sequence (vocabulary slices)
constexpr int kST = 256;      // threads per CTA
constexpr int kSW = kST / 32;
constexpr int kSMaxK = 16;    // drafted tokens per sequence served here
constexpr int kSRows = 2 * kSMaxK + 1;
constexpr size_t kSSmem = 200 * 1024;

enum { QS_LOGITS = 0, QS_PROBS_T1 = 1, QS_PROBS_T = 2 };

struct __align__(16) SmallSh {
  uint64_t bar;
  float2 part[kSRows][kSC];    // every CTA's (max, sum) per row (replicated)
  float2 wpart[kSRows][kSW];   // this CTA's per-warp partials
  float2 xab[kSMaxK][kSC];     // rank 0: every CTA's (alpha, residual mass)
  float2 xpq[kSMaxK];          // rank 0: p and q at the drafted tokens
  uint32_t xbits[kSC];         // rank 0: every CTA's status bits so far
  float Lp[kSMaxK + 1], Lq[kSMaxK], invZq[kSMaxK];
  float wtot[kSW];
  int dec_owner, dec_sel, dec_n, dec_mode;  // from rank 0
  float dec_t;
  uint32_t dec_bits;
  int pick_thread;
  uint32_t cta_bits;
};

__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
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
// eight consecutive elements from shared memory (16-byte aligned)
template <typename T>
__device__ __forceinline__ void ld8s(const T* p, float v[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x);
    v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z);
    v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
  } else {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}
// online (max, sum 2^(v - max)) over eight more values
__device__ __forceinline__ void online8(const float v[8], float& m, float& z) {
  float mx = v[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, v[i]);
  if (mx > m) {
    z = (m == neg_inf()) ? 0.f : z * ex2(m - mx);
    m = mx;
  }
  if (m != neg_inf()) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      s0 += ex2(v[i] - m);
      s1 += ex2(v[i + 1] - m);
    }
    z += s0 + s1;
  }
}
// draft probability from the draft row's element y and its normaliser
template <int QK>
__device__ __forceinline__ float q_of(float y, float kt, float invT, float nLq, float iZ) {
  if constexpr (QK == QS_LOGITS) return ex2(fmaf(y, kt, nLq));
  else if constexpr (QK == QS_PROBS_T1) return __fmul_rn(y, iZ);
  else return ex2(fmaf(lg2(y), invT, nLq));
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
  // this warp's part of the slice (whole groups of 8 logits)
  const int sub = (len + kSW * 8 - 1) / (kSW * 8) * 8;
  const int s0 = min(len, w * sub), s1 = min(len, s0 + sub);
  uint32_t bits = 0;

  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
    sh.cta_bits = 0;
  }
  cluster_arrive_relaxed();
  __syncthreads();
  if (tid == 0 && len > 0) {
    const uint32_t bt = (uint32_t)len * sizeof(TT), bd = (uint32_t)len * sizeof(TD);
    mbar_expect_tx(&sh.bar, (uint32_t)(K + 1) * bt + (uint32_t)K * bd);
    const TT* tg = reinterpret_cast<const TT*>(a.target);
    const TD* dg = reinterpret_cast<const TD*>(a.draft);
    for (int r = 0; r <= K; ++r)
      bulk_g2s(const_cast<TT*>(tsm) + (size_t)r * slice,
               tg + ((int64_t)b * (K + 1) + r) * V + r0, bt, &sh.bar);
    for (int k = 0; k < K; ++k)
      bulk_g2s(const_cast<TD*>(dsm) + (size_t)k * slice, dg + ((int64_t)b * K + k) * V + r0, bd,
               &sh.bar);
  }
  if (len > 0 && !mbar_wait_bounded(&sh.bar, 0)) bits |= SPEC_STATUS_TIMEOUT;

  // 1. (max, sum) of every row over this warp's part, then over the CTA,
  //    broadcast into every CTA of the cluster
  for (int r = 0; r < nrows; ++r) {
    float m = neg_inf(), z = 0.f;
    const bool plain = QK == QS_PROBS_T1 && r > K;
    if (r <= K) {
      const TT* row = tsm + (size_t)r * slice;
      for (int e = s0 + lane * 8; e < s1; e += 256) {
        float v[8];
        ld8s(row + e, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], kt);
        online8(v, m, z);
      }
    } else {
      const TD* row = dsm + (size_t)(r - K - 1) * slice;
      for (int e = s0 + lane * 8; e < s1; e += 256) {
        float v[8];
        ld8s(row + e, v);
        if constexpr (QK == QS_PROBS_T1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) z += v[i];
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[i] = QK == QS_LOGITS ? __fmul_rn(v[i], kt) : __fmul_rn(lg2(v[i]), invT);
          online8(v, m, z);
        }
      }
    }
    MaxSum A;
    if (plain) A = MaxSum{0.f, warp_sum(z)};
    else A = warp_ms(MaxSum{m, z});
    if (lane == 0) sh.wpart[r][w] = make_float2(A.m, A.z);
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started
  if (tid < nrows) {
    const bool plain = QK == QS_PROBS_T1 && tid > K;
    MaxSum A = plain ? MaxSum{0.f, 0.f} : MaxSum{neg_inf(), 0.f};
    for (int k = 0; k < kSW; ++k) {
      const float2 v = sh.wpart[tid][k];
      if (plain) A.z += v.y;
      else A = ms_combine(A, MaxSum{v.x, v.y});
    }
    const uint32_t dst = smem_u32(&sh.part[tid][rank]);
    for (uint32_t c = 0; c < kSC; ++c) st_dsmem_f32x2(mapa(dst, c), make_float2(A.m, A.z));
  }
  cluster_sync();
  if (tid < nrows) {
    const int r = tid;
    const bool plain = QK == QS_PROBS_T1 && r > K;
    MaxSum A = plain ? MaxSum{0.f, 0.f} : MaxSum{neg_inf(), 0.f};
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

  // 2. acceptance mass and residual mass of every drafted row; p and q at the
  //    drafted token from the CTA whose slice holds it
  for (int k = 0; k < K; ++k) {
    const TT* tr = tsm + (size_t)k * slice;
    const TD* dr = dsm + (size_t)k * slice;
    const float nLp = -sh.Lp[k], nLq = -sh.Lq[k], iZ = sh.invZq[k];
    float al = 0.f, rl = 0.f;
    for (int e = s0 + lane * 8; e < s1; e += 256) {
      float x[8], y[8];
      ld8s(tr + e, x);
      ld8s(dr + e, y);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = ex2(fmaf(x[i], kt, nLp));
        const float mn = fminf(p, q_of<QK>(y[i], kt, invT, nLq, iZ));
        al += mn;
        rl += p - mn;
      }
    }
    al = warp_sum(al);
    rl = warp_sum(rl);
    if (lane == 0) sh.wpart[k][w] = make_float2(al, rl);
  }
  __syncthreads();
  if (tid < K) {
    const int k = tid;
    float A = 0.f, Rm = 0.f;
    for (int c = 0; c < kSW; ++c) {
      A += sh.wpart[k][c].x;
      Rm += sh.wpart[k][c].y;
    }
    st_dsmem_f32x2(at_rank(&sh.xab[k][rank], 0), make_float2(A, Rm));
    const int x = a.node_tokens[(int64_t)b * K + k];
    if (x >= r0 && x < r0 + len) {
      const float px = ex2(fmaf(elem(tsm + (size_t)k * slice, x - r0), kt, -sh.Lp[k]));
      const float qx = q_of<QK>(elem(dsm + (size_t)k * slice, x - r0), kt, invT, -sh.Lq[k],
                                sh.invZq[k]);
      st_dsmem_f32x2(at_rank(&sh.xpq[k], 0), make_float2(px, qx));
    }
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits) atomicOr(&sh.cta_bits, bits);
  __syncthreads();
  if (tid == 0) st_dsmem_u32(at_rank(&sh.xbits[rank], 0), sh.cta_bits);
  cluster_sync();

  // 3. decisions, outputs and the slice of the draw (rank 0)
  if (rank == 0 && tid == 0) {
    uint32_t all = 0;
    for (int c = 0; c < kSC; ++c) all |= sh.xbits[c];
    const uint64_t seed = a.prm.seed;
    const uint32_t off = a.prm.philox_offset;
    for (int k = 0; k < K; ++k) {
      float A = 0.f;
      for (int c = 0; c < kSC; ++c) A += sh.xab[k][c].x;
      a.mass[(int64_t)b * K + k] = A;
    }
    int n = K;
    for (int k = 0; k < K && n == K; ++k) {
      const int x = a.node_tokens[(int64_t)b * K + k];
      bool acc;
      if (x < 0 || x >= V) {
        all |= SPEC_STATUS_TOKEN_RANGE;
        acc = false;
      } else {
        const float px = sh.xpq[k].x, qx = sh.xpq[k].y;
        if (qx == 0.f) {
          all |= SPEC_STATUS_QZERO_ACCEPT;
          acc = true;
        } else {
          acc = philox_uniform(seed, off, (uint32_t)b, (uint32_t)k, 0) < px / qx;
        }
        // a rejected token leaves the draft without its mass: none left
        if (!acc && !(1.f - qx > 0.f)) all |= SPEC_STATUS_DRAFT_EXHAUSTED;
      }
      if (!acc) n = k;
    }
    // the draw's weights: residual of row n, else p of row n (no residual
    // mass, flagged) or of row K (every draft accepted)
    int mode = 1;
    if (n < K) {
      float Rm = 0.f;
      for (int c = 0; c < kSC; ++c) Rm += sh.xab[n][c].y;
      if (Rm > 0.f) mode = 0;
      else all |= SPEC_STATUS_RESIDUAL_ZERO;
    }
    float wc[kSC], tot = 0.f;
#pragma unroll
    for (int c = 0; c < kSC; ++c) {
      if (mode == 0) {
        wc[c] = sh.xab[n][c].y;
      } else {
        const float2 v = sh.part[n][c];
        wc[c] = v.x == neg_inf() ? 0.f : v.y * ex2(v.x - sh.Lp[n]);
      }
      tot += wc[c];
    }
    const float u = philox_uniform(seed, off, (uint32_t)b, (uint32_t)n, 1);
    float t = u * tot, run = 0.f;
    int sel = -1, last = -1;
#pragma unroll
    for (int c = 0; c < kSC; ++c) {
      if (wc[c] > 0.f) {
        last = c;
        if (sel < 0 && run + wc[c] > t) sel = c;
      }
      if (sel < 0) run += wc[c];
    }
    if (sel < 0 && last >= 0) {  // rounding: the last slice with mass, its last token
      sel = last;
      t = 3.0e38f;
      run = 0.f;
      all |= SPEC_STATUS_CDF_FALLBACK;
    }
    a.count[b] = n;
    int32_t* out = a.out_tokens + (int64_t)b * (K + 1);
    for (int k = 0; k < n; ++k) out[k] = a.node_tokens[(int64_t)b * K + k];
    for (int k = n + 1; k <= K; ++k) out[k] = -1;
    if (sel < 0) out[n] = 0;  // no mass anywhere (NaN rows, flagged)
    const int owner = sel < 0 ? 0 : sel;
    for (uint32_t c = 0; c < kSC; ++c) {
      st_dsmem_u32(at_rank(&sh.dec_owner, c), (uint32_t)owner);
      st_dsmem_u32(at_rank(&sh.dec_sel, c), (uint32_t)sel);
      st_dsmem_u32(at_rank(&sh.dec_n, c), (uint32_t)n);
      st_dsmem_u32(at_rank(&sh.dec_mode, c), (uint32_t)mode);
      st_dsmem_f32(at_rank(&sh.dec_t, c), t - run);
      st_dsmem_u32(at_rank(&sh.dec_bits, c), all);
    }
  }
  cluster_sync();  // the last cluster barrier: no peer touches this CTA after it
  if (sh.dec_owner != (int)rank) return;

  // 4. inverse CDF inside the owning slice, in vocabulary order: the first
  //    thread whose range passes the remaining threshold, then its element
  const int n = sh.dec_n, mode = sh.dec_mode;
  if (tid == 0) sh.cta_bits = 0;
  if (sh.dec_sel >= 0) {
    const TT* tr = tsm + (size_t)n * slice;
    const TD* dr = dsm + (size_t)(n < K ? n : 0) * slice;
    const float nLp = -sh.Lp[n];
    const float nLq = n < K ? -sh.Lq[n] : 0.f, iZ = n < K ? sh.invZq[n] : 0.f;
    auto wgt = [&](int i) -> float {
      const float p = ex2(fmaf(elem(tr, i), kt, nLp));
      return mode == 0 ? fmaxf(0.f, p - q_of<QK>(elem(dr, i), kt, invT, nLq, iZ)) : p;
    };
    const int per = (len + kST - 1) / kST;
    const int i0 = min(len, tid * per), i1 = min(len, i0 + per);
    float mine = 0.f;
    for (int i = i0; i < i1; ++i) mine += wgt(i);
    float inc = mine;  // inclusive scan over the CTA's threads, in order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sh.wtot[w] = inc;
    if (tid == 0) sh.pick_thread = kST;
    __syncthreads();
    float before = 0.f;
    for (int k = 0; k < w; ++k) before += sh.wtot[k];
    inc += before;
    const float tl = sh.dec_t;
    if (mine > 0.f && inc > tl) atomicMin(&sh.pick_thread, tid);
    __syncthreads();
    int pt = sh.pick_thread;
    bool fallback = false;
    if (pt == kST) {  // rounding: the last thread with mass
      __syncthreads();
      if (tid == 0) sh.pick_thread = -1;
      __syncthreads();
      if (mine > 0.f) atomicMax(&sh.pick_thread, tid);
      __syncthreads();
      pt = sh.pick_thread;
      fallback = true;
    }
    if (tid == pt) {
      const float tt = fallback ? 3.0e38f : tl - (inc - mine);
      float c = 0.f;
      int pick = -1, lastp = -1;
      for (int i = i0; i < i1; ++i) {
        const float wv = wgt(i);
        c += wv;
        if (wv > 0.f) {
          lastp = i;
          if (c > tt) {
            pick = i;
            break;
          }
        }
      }
      if (pick < 0) {
        pick = lastp;
        atomicOr(&sh.cta_bits, SPEC_STATUS_CDF_FALLBACK);
      }
      a.out_tokens[(int64_t)b * (K + 1) + n] = r0 + (pick < 0 ? 0 : pick);
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
