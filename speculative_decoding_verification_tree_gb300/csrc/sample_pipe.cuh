// Pipelined sampled verification (temperature > 0, full vocabulary), the
// bandwidth path for rows up to 131072 logits.
//
// Same method as unit_full in sample_full.cu (accept test u < p'(x)/q'(x),
// residual max(0, p - C q), inverse-CDF draw in vocabulary order), organised
// for HBM streaming on GB300:
//  * row_meta (a small kernel ahead of it) writes one record per row: draft
//    row, children in index order with their tokens, the target / draft
//    logits at those tokens, and the row's Philox uniforms -- so the
//    streaming kernel issues no dependent global loads and no Philox rounds;
//  * persistent thread-block clusters, one 512-thread CTA per SM; each CTA of
//    a cluster owns one contiguous vocabulary slice of every row the cluster
//    verifies; one loader thread keeps S shared-memory stages in flight with
//    TMA bulk copies of the next rows' slices and records, issued while its
//    warp waits for a cluster exchange anyway;
//  * all 16 warps copy a landed slice into registers (up to 32 logits of each
//    row per thread), the stage is refilled at once, and every pass runs out
//    of registers: base-2 exps relative to the thread max (kept, so pass B
//    rescales instead of recomputing them), then alpha, max(0, p - q) and p;
//  * CTA reductions are warp-0 shuffle trees; cluster statistics travel as
//    16-byte st.async stores from warp 0's registers into every peer's shared
//    memory, completing transaction bytes on the peer's mbarrier, and every
//    warp combines the received statistics itself (same shuffle order in all
//    CTAs) -- no cluster barrier and no extra CTA barrier per exchange;
//  * a second exchange happens only after a rejected child; a leaf's bonus
//    draw needs nothing beyond the first (the per-rank mass of p follows from
//    the statistics);
//  * alpha leaves as per-CTA partials, summed in rank order by the walk.
#pragma once

#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace pipe {
namespace {  // internal to each translation unit that instantiates it

constexpr int kCW = 16;                 // warps
constexpr int kCT = kCW * 32;           // threads
constexpr int kThreads = kCT;
constexpr int kTile = 128;              // elements per warp per tile
constexpr int kMaxC = 8;
constexpr int kMaxStages = 4;
constexpr int kMaxKids = SPEC_MAX_CHILDREN;
constexpr int kBar = 1;                 // named barrier id

enum QKind { Q_LOGITS = 0, Q_PROBS_T1 = 1, Q_PROBS_T = 2 };

using Params = ::sv::PipeParams;  // slice = kCW * (EPT / 4) * kTile elements

// Per-row record built by row_meta.  Global layout (stride rec_bytes):
// header, kid[kidcap], then kidcap floats of accept uniforms.  It is copied
// byte for byte to the start of a shared-memory Meta, so the uniforms of a
// record with kidcap slots start at &kid[kidcap].
struct Kid {
  int node;     // drafted node index
  int tok;      // its token
  float raw_t;  // target logit at the token
  float raw_q;  // draft logit / probability at the token
};
struct __align__(16) Meta {
  int qr;          // draft row index within the sequence, or -1
  int nk;          // children (capped at kidcap)
  uint32_t bad;    // status bits found while building the record
  float u_draw;    // u(b, r, 1): the row's replacement / bonus draw
  Kid kid[kMaxKids];
  float uspace[kMaxKids];
};

static_assert(sizeof(Meta) == 16 + 20 * kMaxKids, "record layout");

template <typename TT, typename TD>
__global__ void __launch_bounds__(256) row_meta(VerifyShape s, VerifyArgs a, int kidcap,
                                                int rec_bytes) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (unit >= s.rows()) return;
  const int n = s.n, V = s.V;
  const int b = (int)(unit / (n + 1));
  const int r = (int)(unit - (int64_t)b * (n + 1));
  uint32_t bad = 0;
  int qr = -1;
  if (s.chain) {
    qr = (r < n) ? r : -1;
  } else if (a.q_row) {
    qr = a.q_row[unit];
    if (qr < -1 || qr >= s.R) {
      bad |= SPEC_STATUS_BAD_TREE;
      qr = -1;
    }
  }
  const TT* trow = reinterpret_cast<const TT*>(a.target) + unit * (int64_t)V;
  const TD* drow =
      qr >= 0 ? reinterpret_cast<const TD*>(a.draft) + ((int64_t)b * s.R + qr) * V : nullptr;
  unsigned char* recb = a.meta + unit * (int64_t)rec_bytes;
  Kid* kids = reinterpret_cast<Kid*>(recb + 16);
  float* ukid = reinterpret_cast<float*>(recb + 16 + 16 * kidcap);
  auto put = [&](int pos, int node, int tok) {
    float rt = 0.f, rq = 0.f;
    if (tok >= 0 && tok < V) {
      rt = ElemIO<TT>::get(trow, tok);
      rq = drow ? ElemIO<TD>::get(drow, tok) : 0.f;
    }
    kids[pos] = Kid{node, tok, rt, rq};
    ukid[pos] = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b, (uint32_t)node, 0u);
  };
  int cnt = 0;
  if (s.chain) {
    if (r < n) {
      cnt = 1;
      if (lane == 0) put(0, r, a.node_tokens[(int64_t)b * n + r]);
    }
  } else {
    const int32_t* par = a.parent + (int64_t)b * n;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int j = j0 + lane;
      const int p = (j < n) ? par[j] : -2;
      const bool valid = (p >= -1 && p < j);
      if (j < n && !valid) bad |= SPEC_STATUS_BAD_TREE;
      const uint32_t m = __ballot_sync(0xffffffffu, j < n && valid && p == r - 1);
      if (m & (1u << lane)) {
        const int pos = cnt + __popc(m & ((1u << lane) - 1));
        if (pos < kidcap) put(pos, j, a.node_tokens[(int64_t)b * n + j]);
        else bad |= SPEC_STATUS_BAD_TREE;
      }
      cnt += __popc(m);
    }
    cnt = min(cnt, kidcap);
  }
  if (cnt > 0 && qr < 0) {
    bad |= SPEC_STATUS_BAD_TREE;
    cnt = 0;
  }
  bad = __reduce_or_sync(0xffffffffu, bad);
  if (lane == 0) {
    Meta* h = reinterpret_cast<Meta*>(recb);
    h->qr = qr;
    h->nk = cnt;
    h->bad = bad;
    h->u_draw = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b, (uint32_t)r, 1u);
    a.qres[unit] = qr;
  }
}

struct Smem {
  uint64_t full[kMaxStages];
  uint64_t mfull[3];
  uint64_t xbar[2];
  float4 xslot[2][kMaxC];   // incoming per-rank payloads (two in flight)
  Meta meta[3];
  float4 wred[kCW];         // per-warp partials
  float wr[kCW], wp[kCW], wx[2][kCW];
  float rk_p[kMaxC], rk_r[kMaxC], rkx[2][kMaxC];
  float4 bc;                // warp 0 -> all
  int ibc[4];
  int qring[4];             // draft rows of upcoming refills (loop index & 3)
};

__device__ __forceinline__ float resid_w(float p, float q, float C) {
  return C == 0.f ? p : fmaxf(0.f, fmaf(-C, q, p));
}

template <typename T>
__device__ __forceinline__ T pad_logit();
template <>
__device__ __forceinline__ float pad_logit<float>() { return neg_inf(); }
template <>
__device__ __forceinline__ uint16_t pad_logit<uint16_t>() { return (uint16_t)0xff80u; }

// Warp-wide sum with a fixed tree (identical in every warp and CTA).
__device__ __forceinline__ float tree_sum(float v) { return warp_sum(v); }

// Exchange number xq: lanes 0..C-1 of warp 0 push `mine` to every CTA of the
// cluster (lane k -> CTA k); every thread then waits for the C payloads of
// this exchange in sm.xslot[xq & 1].  Only warp 0 may call with real data;
// the other warps only wait.
__device__ __forceinline__ void exchange(Smem& sm, int xq, int C, uint32_t rank, int warp,
                                         int lane, float4 mine, uint32_t* status) {
  const int sl = xq & 1;
  if (warp == 0) {
    if (lane == 0) mbar_expect_tx(&sm.xbar[sl], (uint32_t)C * 16u);
    if (lane < C) {
      const uint32_t slot = mapa(smem_u32(&sm.xslot[sl][rank]), (uint32_t)lane);
      const uint32_t bar = mapa(smem_u32(&sm.xbar[sl]), (uint32_t)lane);
      st_async_v4(slot, mine, bar);
    }
  }
  if (!mbar_wait_cluster_bounded(&sm.xbar[sl], (uint32_t)((xq >> 1) & 1)))
    flag_status(status, SPEC_STATUS_TIMEOUT);
}

template <typename TT, typename TD, int QK, int EPT>
__global__ void __launch_bounds__(kThreads, 1) unit_pipe(Params P) {
  constexpr int kTPW = EPT / 4;  // tiles per warp
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  const VerifyShape& s = P.s;
  const VerifyArgs& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int C = (int)cluster_nctarank();
  const int cid = blockIdx.x / C;
  const int ncl = P.nclusters;
  const int n = s.n;
  const int64_t nunits = s.rows();
  const int V = s.V;
  const int slice = P.slice;
  const int S = P.stages;
  const int s0 = (int)rank * slice;
  const int len = max(0, min(slice, V - s0));
  const size_t tbytes = (size_t)slice * sizeof(TT);
  const size_t stage_bytes = tbytes + (size_t)slice * sizeof(TD);
  auto stage_t = [&](int st) { return reinterpret_cast<TT*>(dyn + st * stage_bytes); };
  auto stage_d = [&](int st) { return reinterpret_cast<TD*>(dyn + st * stage_bytes + tbytes); };

  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&sm.full[i], 1);
    for (int i = 0; i < 3; ++i) mbar_init(&sm.mfull[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.xbar[i], 1);
    }
    fence_mbar_init();
  }
  // the part of each stage past the row end never changes: pad it once
  for (int st = 0; st < S; ++st) {
    TT* tb = stage_t(st);
    TD* db = stage_d(st);
    for (int i = len + tid; i < slice; i += kThreads) {
      tb[i] = pad_logit<TT>();
      db[i] = (QK == Q_LOGITS) ? pad_logit<TD>() : (TD)0;
    }
  }
  cluster_sync();  // every CTA's barriers exist before the first st.async

  auto issue_slices = [&](int64_t u, int q, int stg) {
    const int bb = (int)(u / (n + 1));
    const TT* trow = reinterpret_cast<const TT*>(a.target) + u * (int64_t)V;
    const uint32_t tb = (uint32_t)len * sizeof(TT);
    const uint32_t db = q >= 0 ? (uint32_t)len * sizeof(TD) : 0u;
    mbar_expect_tx(&sm.full[stg], tb + db);
    if (tb) bulk_g2s(stage_t(stg), trow + s0, tb, &sm.full[stg]);
    if (db) {
      const TD* drow = reinterpret_cast<const TD*>(a.draft) + ((int64_t)bb * s.R + q) * V;
      bulk_g2s(stage_d(stg), drow + s0, db, &sm.full[stg]);
    }
  };
  auto issue_meta = [&](int64_t u, int buf) {
    mbar_expect_tx(&sm.mfull[buf], (uint32_t)P.rec_bytes);
    bulk_g2s(&sm.meta[buf], a.meta + u * (int64_t)P.rec_bytes, (uint32_t)P.rec_bytes,
             &sm.mfull[buf]);
  };
  // The loader thread (lane 0 of the last warp) issues every bulk copy, and
  // does so while its warp waits for the first cluster exchange of a row, so
  // no warp ever waits behind a copy being issued.  Row j's slices refill
  // stage j % S (freed when row j - S was copied into registers); its record
  // goes to buffer j % 3 (freed when row j - 3 finished).  The draft row of
  // row j is loaded two rows before it is needed (qring).
  auto q_of_index = [&](int j) -> int {
    const int64_t u = cid + (int64_t)j * ncl;
    return (u < nunits) ? a.qres[u] : -1;
  };
  const bool ldr = (tid == kCT - 32);
  if (ldr) {
    for (int i = 0; i < S; ++i) {
      const int64_t u = cid + (int64_t)i * ncl;
      if (u < nunits) issue_slices(u, a.qres[u], i);
    }
    for (int i = 0; i < 2; ++i) {
      const int64_t u = cid + (int64_t)i * ncl;
      if (u < nunits) issue_meta(u, i);
      sm.qring[(S + i) & 3] = q_of_index(S + i);
    }
  }

  int xq = 0;
  for (int it = 0;; ++it) {
    const int64_t unit = cid + (int64_t)it * ncl;
    if (unit >= nunits) break;
    const int st = it % S, mb = it % 3;
    const int64_t u_pre = unit + (int64_t)S * ncl;  // refills stage st
    const int64_t u_meta = unit + 2 * (int64_t)ncl;  // record into (it + 2) % 3
    const int q_later = ldr ? q_of_index(it + S + 2) : -1;
    bool ok = mbar_wait_bounded(&sm.full[st], (uint32_t)((it / S) & 1));
    ok &= mbar_wait_bounded(&sm.mfull[mb], (uint32_t)((it / 3) & 1));
    if (!ok) flag_status(a.status, SPEC_STATUS_TIMEOUT);
    const Meta& M = sm.meta[mb];
    const bool has_q = M.qr >= 0;
    const int nk = M.nk;

    // slice -> registers
    float ep[EPT], eq[EPT];
    {
      const TT* tb = stage_t(st);
      const TD* db = stage_d(st);
#pragma unroll
      for (int t = 0; t < kTPW; ++t) {
        const int e = (warp * kTPW + t) * kTile + lane * 4;
        ElemIO<TT>::get4(tb + e, &ep[4 * t]);
        if (has_q) {
          ElemIO<TD>::get4(db + e, &eq[4 * t]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) eq[4 * t + j] = 0.f;
        }
      }
    }

    // pass A: thread max, then base-2 exps relative to it (kept)
    float mt = neg_inf();
#pragma unroll
    for (int j = 0; j < EPT; ++j) mt = fmaxf(mt, __fmul_rn(ep[j], P.kt));
    float zt = 0.f;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      ep[j] = (mt == neg_inf()) ? 0.f : ex2(fmaf(ep[j], P.kt, -mt));
      zt += ep[j];
    }
    float mq = neg_inf(), zq = 0.f;
    if (has_q) {
      if constexpr (QK == Q_PROBS_T1) {
#pragma unroll
        for (int j = 0; j < EPT; ++j) zq += eq[j];
      } else {
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          const float sq = (QK == Q_LOGITS) ? __fmul_rn(eq[j], P.kt) : __fmul_rn(lg2(eq[j]), P.invT);
          eq[j] = sq;
          mq = fmaxf(mq, sq);
        }
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          eq[j] = (mq == neg_inf()) ? 0.f : ex2(eq[j] - mq);
          zq += eq[j];
        }
      }
    }
    {
      const MaxSum A = warp_ms(MaxSum{mt, zt});
      float m2 = 0.f, z2;
      if (QK == Q_PROBS_T1) {
        z2 = warp_sum(zq);
      } else {
        const MaxSum Bq = warp_ms(MaxSum{mq, zq});
        m2 = Bq.m;
        z2 = Bq.z;
      }
      if (lane == 0) sm.wred[warp] = make_float4(A.m, A.z, m2, z2);
    }
    named_sync(kBar, kCT);  // partials ready; every thread is done with stage st
    if (ldr) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (u_pre < nunits) issue_slices(u_pre, sm.qring[(it + S) & 3], st);
      if (u_meta < nunits) issue_meta(u_meta, (it + 2) % 3);
      sm.qring[(it + S + 2) & 3] = q_later;
    }
    // CTA statistics (warp 0, 16-lane tree) -> exchange 1
    {
      float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
      if (warp == 0) {
        const float4 v = (lane < kCW) ? sm.wred[lane] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
        MaxSum A{v.x, v.y}, Bq{v.z, v.w};
        float z1 = (lane < kCW) ? v.w : 0.f;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          A = ms_combine(A, MaxSum{__shfl_xor_sync(0xffffffffu, A.m, o),
                                   __shfl_xor_sync(0xffffffffu, A.z, o)});
          if (QK == Q_PROBS_T1) {
            z1 += __shfl_xor_sync(0xffffffffu, z1, o);
          } else {
            Bq = ms_combine(Bq, MaxSum{__shfl_xor_sync(0xffffffffu, Bq.m, o),
                                       __shfl_xor_sync(0xffffffffu, Bq.z, o)});
          }
        }
        A.m = __shfl_sync(0xffffffffu, A.m, 0);
        A.z = __shfl_sync(0xffffffffu, A.z, 0);
        z1 = __shfl_sync(0xffffffffu, z1, 0);
        Bq.m = __shfl_sync(0xffffffffu, Bq.m, 0);
        Bq.z = __shfl_sync(0xffffffffu, Bq.z, 0);
        mine = make_float4(A.m, A.z, QK == Q_PROBS_T1 ? 0.f : Bq.m, QK == Q_PROBS_T1 ? z1 : Bq.z);
      }
      exchange(sm, xq, C, rank, warp, lane, mine, a.status);
    }
    // cluster statistics: every warp combines the C payloads (8-lane tree)
    float Lp, Lq = 0.f, invZq = 0.f, zq_tot = 0.f, zp_tot;
    {
      const float4* xs = sm.xslot[xq & 1];
      const float4 v = (lane < C) ? xs[lane] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
      MaxSum A{v.x, v.y}, Bq{v.z, v.w};
      float z1 = (lane < C) ? v.w : 0.f;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        A = ms_combine(A, MaxSum{__shfl_xor_sync(0xffffffffu, A.m, o),
                                 __shfl_xor_sync(0xffffffffu, A.z, o)});
        if (QK == Q_PROBS_T1) {
          z1 += __shfl_xor_sync(0xffffffffu, z1, o);
        } else {
          Bq = ms_combine(Bq, MaxSum{__shfl_xor_sync(0xffffffffu, Bq.m, o),
                                     __shfl_xor_sync(0xffffffffu, Bq.z, o)});
        }
      }
      A.m = __shfl_sync(0xffffffffu, A.m, 0);
      A.z = __shfl_sync(0xffffffffu, A.z, 0);
      z1 = __shfl_sync(0xffffffffu, z1, 0);
      Bq.m = __shfl_sync(0xffffffffu, Bq.m, 0);
      Bq.z = __shfl_sync(0xffffffffu, Bq.z, 0);
      Lp = A.m + log2f(A.z);
      zp_tot = A.z;
      if (has_q) {
        if (QK == Q_PROBS_T1) {
          invZq = 1.f / z1;
          zq_tot = z1;
        } else {
          Lq = Bq.m + log2f(Bq.z);
          zq_tot = Bq.z;
        }
      }
      // per-rank mass of p (bonus draw) from the statistics
      if (warp == 0 && lane < C) sm.rk_p[lane] = (v.y > 0.f) ? v.y * ex2(v.x - Lp) : 0.f;
    }
    ++xq;

    // pass B: p, q in place; alpha, max(0, p - q) and p per warp
    {
      const float sp = (mt == neg_inf()) ? 0.f : ex2(mt - Lp);
      const float sq = (QK == Q_PROBS_T1) ? invZq : ((mq == neg_inf()) ? 0.f : ex2(mq - Lq));
      // sum of p: only a row without children draws from p (bonus); the
      // rare zero-residual fallback of a row with children recomputes it
      float acc_a = 0.f, acc_r = 0.f, acc_p = 0.f;
      if (has_q) {
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          const float p = ep[j] * sp;
          const float q = eq[j] * sq;
          ep[j] = p;
          eq[j] = q;
          const float mn = fminf(p, q);
          acc_a += mn;
          acc_r += p - mn;
        }
        if (nk == 0) {
#pragma unroll
          for (int j = 0; j < EPT; ++j) acc_p += ep[j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          ep[j] *= sp;
          acc_p += ep[j];
        }
      }
      acc_a = warp_sum(acc_a);
      acc_r = warp_sum(acc_r);
      acc_p = warp_sum(acc_p);
      if (lane == 0) {
        sm.wred[warp].x = acc_a;
        sm.wr[warp] = acc_r;
        sm.wp[warp] = acc_p;
      }
    }
    named_sync(kBar, kCT);
    const float negLp = -Lp, negLq = -Lq;
    auto q_point = [&](float raw) -> float {
      if constexpr (QK == Q_LOGITS) return ex2(fmaf(raw, P.kt, negLq));
      else if constexpr (QK == Q_PROBS_T1) return __fmul_rn(raw, invZq);
      else return ex2(fmaf(lg2(raw), P.invT, negLq));
    };
    // warp 0: alpha partial, CTA residual mass, first child's decision
    float Rcta = 0.f;
    if (warp == 0) {
      float va = (lane < kCW) ? sm.wred[lane].x : 0.f;
      float vr = (lane < kCW) ? sm.wr[lane] : 0.f;
      va = warp_sum(va);
      vr = warp_sum(vr);
      Rcta = vr;
      if (lane == 0) {
        if (has_q) a.alpha_part[unit * kMaxC + rank] = va;
        if (rank == 0) {
          uint32_t bad = M.bad;
          if (!(zp_tot > 0.f) || isnan(zp_tot)) bad |= SPEC_STATUS_NAN;
          if (has_q && !(zq_tot > 0.f)) bad |= SPEC_STATUS_NAN;
          flag_status(a.status, bad);
        }
      }
    }

    // sibling recursion (cluster-uniform control flow); decisions by lane 0
    // of warp 0 from the record's point logits and uniforms
    const float* ukid = reinterpret_cast<const float*>(&M.kid[P.kidcap]);
    float Cc = 0.f, W = 1.f, D = 1.f;
    int accepted = -1;
    int src = 0, xb = 0;
    uint32_t st_bits = 0;
    for (int k = 0; k < nk; ++k) {
      if (tid == 0) {
        const int x = M.kid[k].tok;
        int dec = 0;
        if (x < 0 || x >= V) {
          st_bits |= SPEC_STATUS_TOKEN_RANGE;
        } else {
          bool removed = false;
          for (int i = 0; i < k; ++i) removed |= (M.kid[i].tok == x);
          const float pv = ex2(fmaf(M.kid[k].raw_t, P.kt, negLp));
          const float qv = q_point(M.kid[k].raw_q);
          const float ax = resid_w(pv, qv, Cc);
          const float qj = removed ? 0.f : qv / D;
          if (qj == 0.f) {
            dec = 1;
            st_bits |= SPEC_STATUS_QZERO_ACCEPT;
          } else {
            dec = (ukid[k] < (ax / W) / qj) ? 1 : 0;
          }
        }
        sm.ibc[0] = dec;
        sm.bc.x = Cc + W / D;
      }
      named_sync(kBar, kCT);
      const int dec = sm.ibc[0];
      const float Cn = sm.bc.x;
      if (dec) {
        accepted = M.kid[k].node;
        break;
      }
      float Wn = 0.f;
      int nsrc;
      if (Cc == 0.f && Cn == 1.f) {
        // residual max(0, p - q): per-rank totals by one exchange
        exchange(sm, xq, C, rank, warp, lane, make_float4(Rcta, 0.f, 0.f, 0.f), a.status);
        if (tid == 0) {
          for (int i = 0; i < C; ++i) {
            sm.rk_r[i] = sm.xslot[xq & 1][i].x;
            Wn += sm.rk_r[i];
          }
        }
        ++xq;
        nsrc = 1;
      } else {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc += resid_w(ep[j], eq[j], Cn);
        acc = warp_sum(acc);
        if (lane == 0) sm.wx[xb][warp] = acc;
        named_sync(kBar, kCT);
        float tot = 0.f;
        if (warp == 0) tot = warp_sum((lane < kCW) ? sm.wx[xb][lane] : 0.f);
        exchange(sm, xq, C, rank, warp, lane, make_float4(tot, 0.f, 0.f, 0.f), a.status);
        if (tid == 0) {
          for (int i = 0; i < C; ++i) {
            sm.rkx[xb][i] = sm.xslot[xq & 1][i].x;
            Wn += sm.rkx[xb][i];
          }
        }
        ++xq;
        nsrc = 2 + xb;
      }
      if (tid == 0) {
        int upd = 0;
        if (Wn > 0.f) {
          Cc = Cn;
          W = Wn;
          upd = 1;
        } else {
          st_bits |= SPEC_STATUS_RESIDUAL_ZERO;
        }
        const int x = M.kid[k].tok;
        bool removed = false;
        for (int i = 0; i < k; ++i) removed |= (M.kid[i].tok == x);
        if (x >= 0 && x < V && !removed) D -= q_point(M.kid[k].raw_q);
        if (D <= 0.f) st_bits |= SPEC_STATUS_DRAFT_EXHAUSTED;
        sm.bc = make_float4(Cc, (D <= 0.f) ? 1.f : 0.f, (float)upd, 0.f);
      }
      named_sync(kBar, kCT);
      Cc = sm.bc.x;
      const bool exhausted = sm.bc.y != 0.f;
      if (sm.bc.z != 0.f) {
        src = nsrc;
        if (nsrc >= 2) xb ^= 1;
      }
      named_sync(kBar, kCT);
      if (exhausted) break;
    }

    // draw from p' (leaf: bonus from p) when no child was accepted
    if (accepted < 0) {
      if (src == 0 && nk > 0) {  // fallback to p in a row with children
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc += ep[j];
        acc = warp_sum(acc);
        if (lane == 0) sm.wp[warp] = acc;
        named_sync(kBar, kCT);
      }
      if (warp == 0) {
        // rank: first with running total above t (8-lane inclusive scan)
        const float rkv = (lane < C) ? (src == 0 ? sm.rk_p[lane]
                                                 : (src == 1 ? sm.rk_r[lane] : sm.rkx[src - 2][lane]))
                                     : 0.f;
        float inc = rkv;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const float tot = __shfl_sync(0xffffffffu, inc, 7);
        float t = M.u_draw * tot;
        uint32_t cr = __ballot_sync(0xffffffffu, lane < C && rkv > 0.f && inc > t);
        int sel;
        if (cr) {
          sel = __ffs(cr) - 1;
        } else {  // rounding: last rank with mass, no crossing inside it
          const uint32_t pos = __ballot_sync(0xffffffffu, lane < C && rkv > 0.f);
          sel = pos ? 31 - __clz(pos) : -1;
          t = 3.0e38f;
        }
        const float pre = (sel >= 0) ? __shfl_sync(0xffffffffu, inc - rkv, sel & 31) : 0.f;
        const float tt = t - pre;
        // warp inside the selected CTA (16-lane scan over the per-warp sums)
        int wsel = -1;
        float wpre = 0.f;
        if (sel == (int)rank) {
          const float* wt = src == 0 ? sm.wp : (src == 1 ? sm.wr : sm.wx[src - 2]);
          const float wv = (lane < kCW) ? wt[lane] : 0.f;
          float winc = wv;
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc += y;
          }
          uint32_t wc = __ballot_sync(0xffffffffu, lane < kCW && wv > 0.f && winc > tt);
          if (wc) {
            wsel = __ffs(wc) - 1;
          } else {
            const uint32_t wp2 = __ballot_sync(0xffffffffu, lane < kCW && wv > 0.f);
            wsel = wp2 ? 31 - __clz(wp2) : -1;
          }
          wpre = (wsel >= 0) ? __shfl_sync(0xffffffffu, winc - wv, wsel & 31) : 0.f;
        }
        if (lane == 0) {
          sm.ibc[1] = sel;
          sm.ibc[2] = wsel;
          sm.bc.w = tt - wpre;
          if (sel < 0) {
            st_bits |= SPEC_STATUS_CDF_FALLBACK;
            if (rank == 0) a.row_token[unit] = 0;
          }
        }
      }
      named_sync(kBar, kCT);
      const int sel = sm.ibc[1], wsel = sm.ibc[2];
      if (sel == (int)rank && warp == wsel && wsel >= 0) {
        const float thr = sm.bc.w;
        float run = 0.f;
        int found = -1, lastpos = -1;
#pragma unroll
        for (int t = 0; t < kTPW; ++t) {
          if (found < 0) {
            const int e = (warp * kTPW + t) * kTile + lane * 4;
            float wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) wv[j] = resid_w(ep[4 * t + j], eq[4 * t + j], Cc);
            const float ls = (wv[0] + wv[1]) + (wv[2] + wv[3]);
            float inc = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, inc, o);
              if (lane >= o) inc += y;
            }
            const uint32_t cross = __ballot_sync(0xffffffffu, ls > 0.f && run + inc > thr);
            const uint32_t pos = __ballot_sync(0xffffffffu, ls > 0.f);
            if (pos) {
              const int hl = 31 - __clz(pos);
              int lp = -1;
              if (lane == hl) {
#pragma unroll
                for (int j = 3; j >= 0; --j)
                  if (lp < 0 && wv[j] > 0.f) lp = e + j;
              }
              lastpos = __shfl_sync(0xffffffffu, lp, hl);
            }
            if (cross) {
              const int fl = __ffs(cross) - 1;
              int tok = -1;
              if (lane == fl) {
                float c = run + inc - ls;
                int last = -1;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  if (tok < 0) {
                    if (wv[j] > 0.f) last = e + j;
                    c += wv[j];
                    if (wv[j] > 0.f && c > thr) tok = e + j;
                  }
                }
                if (tok < 0) tok = last;
              }
              found = __shfl_sync(0xffffffffu, tok, fl);
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
          }
        }
        if (lane == 0) {
          int tok = found;
          if (tok < 0) {
            tok = lastpos;
            flag_status(a.status, SPEC_STATUS_CDF_FALLBACK);
          }
          a.row_token[unit] = (tok < 0) ? 0 : s0 + tok;
        }
      }
    }
    if (tid == 0) {
      if (rank == 0) {
        a.row_child[unit] = accepted;
        if (st_bits) flag_status(a.status, st_bits);
      }
    }
    named_sync(kBar, kCT);  // the broadcasts are free again
  }
  cluster_sync();  // no CTA leaves while a peer may still push to it
}

// Walk every sequence along accepted children; reduce alpha partials.
__global__ void pipe_walk(VerifyShape s, VerifyArgs a, int C) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= s.rows()) return;
  const int n = s.n;
  const int b = (int)(row / (n + 1));
  const int r = (int)(row - (int64_t)b * (n + 1));
  bool has_q;
  if (s.chain) {
    has_q = r < n;
  } else {
    const int q = a.q_row ? a.q_row[row] : -1;
    has_q = q >= 0 && q < s.R;
  }
  float m = __int_as_float(0x7fc00000);
  if (has_q) {
    m = 0.f;
    for (int k = 0; k < C; ++k) m += a.alpha_part[row * kMaxC + k];
  }
  if (s.chain) {
    if (r < n) a.mass[(int64_t)b * n + r] = m;
  } else {
    a.mass[row] = m;
  }
  if (r != 0) return;
  const int64_t row0 = row;
  int32_t* out = a.out_tokens + row0;
  int rr = 0, len = 0;
  while (true) {
    const int j = a.row_child[row0 + rr];
    if (j < 0 || j >= n || len >= n) break;
    if (!s.chain) a.path_nodes[(int64_t)b * n + len] = j;
    out[len] = a.node_tokens[(int64_t)b * n + j];
    ++len;
    rr = j + 1;
  }
  out[len] = a.row_token[row0 + rr];
  for (int k = len + 1; k <= n; ++k) out[k] = -1;
  if (!s.chain)
    for (int k = len; k < n; ++k) a.path_nodes[(int64_t)b * n + k] = -1;
  a.count[b] = len;
}

// Geometry: cluster size C, elements per thread EPT and stages for a row of
// V logits; false when the pipelined kernel does not apply.
inline bool geometry(int V, int tsz, int dsz, int* C, int* ept, int* stages, int* slice) {
  const int eptc[3] = {8, 16, 32};
  for (int c = 1; c <= kMaxC; c *= 2) {
    for (int e : eptc) {
      const int sl = kCT * e;  // kCW warps * (e / 4) tiles * 128 elements
      if ((int64_t)c * sl < V) continue;
      const int64_t stage = (int64_t)sl * (tsz + dsz);
      const int ns = (int)((200 * 1024) / stage);
      if (ns < 2) break;
      *C = c;
      *ept = e;
      *stages = ns < kMaxStages ? ns : kMaxStages;
      *slice = sl;
      return true;
    }
  }
  return false;
}

template <typename TT, typename TD, int QK, int EPT>
cudaError_t launch_pipe_t(Params P, int C, cudaStream_t st) {
  auto kern = unit_pipe<TT, TD, QK, EPT>;
  const size_t dyn = (size_t)P.stages * P.slice * (sizeof(TT) + sizeof(TD));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int maxc = 0;
  cfg.gridDim = dim3(C);
  e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (maxc < 1) return cudaErrorInvalidConfiguration;
  const int64_t units = P.s.rows();
  P.nclusters = (int)(units < maxc ? units : maxc);
  row_meta<TT, TD><<<(unsigned)((units + 7) / 8), 256, 0, st>>>(P.s, P.a, P.kidcap, P.rec_bytes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(P.nclusters * C));
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <typename TT, typename TD>
cudaError_t launch_pipe_dt(const Params& P, int C, int ept, int qk, cudaStream_t st) {
#define SV_PIPE_EPT(QK)                                                   \
  if (ept == 8) return launch_pipe_t<TT, TD, QK, 8>(P, C, st);            \
  if (ept == 16) return launch_pipe_t<TT, TD, QK, 16>(P, C, st);          \
  return launch_pipe_t<TT, TD, QK, 32>(P, C, st);
  if (qk == Q_LOGITS) { SV_PIPE_EPT(Q_LOGITS) }
  if (qk == Q_PROBS_T1) { SV_PIPE_EPT(Q_PROBS_T1) }
  SV_PIPE_EPT(Q_PROBS_T)
#undef SV_PIPE_EPT
}

}  // namespace
}  // namespace pipe
}  // namespace sv
