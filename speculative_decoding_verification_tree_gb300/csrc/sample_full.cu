// Sampled verification over the full vocabulary (temperature > 0, no top-k /
// top-p).  One thread-block cluster per tree row ("unit"); each CTA of the
// cluster holds one contiguous vocabulary slice of the row's target logits
// and draft row in shared memory, so every logit is read from HBM exactly once
// while the softmax statistics, the acceptance mass, the sibling recursion and
// the inverse-CDF draw all run out of shared memory.
//
// Method (p = target, q = draft, both softmax(z / T)):
//  * alpha = sum_x min(p, q) ("接受率等于两个分布重叠的质量", "064 · 投机解码").
//  * Children of the row are tried in index order; child j with token x is
//    accepted iff u(b, j, 0) < p'(x) / q'(x) (exactness rule of "投机解码与
//    EAGLE"; q'(x) = 0 accepts, "Bước 1" of the EAGLE-3 lesson).
//  * After a rejection p' <- norm(max(0, p' - q')) (EAGLE-2 notes §2.1; the
//    chain's residual) and x leaves q' (siblings are drafted without
//    replacement).  Unrolled, the unnormalised residual after j rejections is
//    max(0, p - C_j q) with C_j = sum_i W_i / D_i (W_i the residual mass, D_i
//    the q mass left), so each further sibling costs one pass over shared
//    memory and no per-token bookkeeping: a rejected token already has
//    p'(x) < q'(x), so its residual is 0 and stays 0 as C grows.
//  * No child accepted: draw from p' with u(b, r, 1) by inverse CDF in
//    vocabulary order (a leaf: the bonus token from p).
// Per-row outcomes go to the workspace; sampled_walk then follows accepted
// children from the root of every sequence.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kNW = 8;                 // warps per CTA
constexpr int kThreads = kNW * 32;
constexpr int kTile = 128;             // elements per warp step (4 per lane)
constexpr int kSliceQuant = kTile * kNW;
constexpr int kMaxCluster = 8;

enum QKind { Q_LOGITS = 0, Q_PROBS_T1 = 1, Q_PROBS_T = 2 };

struct UnitParams {
  VerifyShape s;
  VerifyArgs a;
  int slice;    // elements per CTA (multiple of kSliceQuant)
  int bulk;     // stage with cp.async.bulk
  float kt;     // log2(e) / T
  float invT;   // 1 / T
};

// Exchange slots read by the other CTAs of the cluster through DSMEM.
struct Xchg {
  float v[4];
};

struct Smem {
  uint64_t bar;
  int nkids;
  int qrow_ok;
  int decision;        // broadcast of thread 0's per-child decision
  int accepted;
  int rank_sel;
  float Lp, Lq, invZq;
  float bc[4];                      // broadcasts from thread 0
  float wp[kNW], wr[kNW];           // per-warp totals of p and max(0, p - q)
  float wx[2][kNW];                 // per-warp totals of two sibling passes
  float rk_p[kMaxCluster];          // per-rank totals of the same
  float rk_r[kMaxCluster];
  float rkx[2][kMaxCluster];
  float red[kNW][4];
  Xchg x[4];                        // 0: stats, 1: pass B, 2/3: sibling passes
  int kid_node[SPEC_MAX_CHILDREN];
  int kid_tok[SPEC_MAX_CHILDREN];
  float kid_p[SPEC_MAX_CHILDREN];
  float kid_q[SPEC_MAX_CHILDREN];
};

template <typename TT, typename TD, int QK>
struct Row {
  const TT* t;  // shared slice of target logits
  const TD* d;  // shared slice of the draft row
  float kt, invT, negLp, negLq, invZq;
  __device__ __forceinline__ float p_of(float raw) const { return ex2(fmaf(raw, kt, negLp)); }
  __device__ __forceinline__ float q_of(float raw) const {
    if constexpr (QK == Q_LOGITS) return ex2(fmaf(raw, kt, negLq));
    else if constexpr (QK == Q_PROBS_T1) return __fmul_rn(raw, invZq);
    else return ex2(fmaf(lg2(raw), invT, negLq));
  }
};

__device__ __forceinline__ float resid_w(float p, float q, float C) {
  return C == 0.f ? p : fmaxf(0.f, fmaf(-C, q, p));
}

// Sum the per-rank slot `slot` component `c` over the cluster in rank order
// and keep the per-rank values.
__device__ __forceinline__ float gather_ranks(Smem& sm, int slot, int c, int C, float* per_rank) {
  float tot = 0.f;
  for (int k = 0; k < C; ++k) {
    const float v = ld_dsmem_f32(mapa(smem_u32(&sm.x[slot].v[c]), (uint32_t)k));
    if (per_rank) per_rank[k] = v;
    tot += v;
  }
  return tot;
}

template <typename TT, typename TD, int QK>
__global__ void __launch_bounds__(kThreads) unit_full(UnitParams P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  const VerifyShape& s = P.s;
  const VerifyArgs& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int C = (int)cluster_nctarank();
  const int64_t unit = blockIdx.x / C;
  const int n = s.n;
  const int b = (int)(unit / (n + 1));
  const int r = (int)(unit - (int64_t)b * (n + 1));
  const int V = s.V;
  const int slice = P.slice;
  TT* tbuf = reinterpret_cast<TT*>(dyn);
  TD* dbuf = reinterpret_cast<TD*>(dyn + (size_t)slice * sizeof(TT));
  const int s0 = (int)rank * slice;
  const int len = max(0, min(slice, V - s0));

  // draft row of this tree row
  int qr = -1;
  if (s.chain) {
    qr = (r < n) ? r : -1;
  } else if (a.q_row) {
    qr = a.q_row[unit];
    if (qr < -1 || qr >= s.R) {
      if (tid == 0 && rank == 0) flag_status(a.status, SPEC_STATUS_BAD_TREE);
      qr = -1;
    }
  }
  const bool has_q = qr >= 0;
  const TT* trow = reinterpret_cast<const TT*>(a.target) + unit * (int64_t)V;
  const TD* drow = has_q ? reinterpret_cast<const TD*>(a.draft) + ((int64_t)b * s.R + qr) * V : nullptr;

  // ---- stage the slice(s) into shared memory
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (P.bulk) {
    if (tid == 0) {
      const uint32_t tb = (uint32_t)len * sizeof(TT);
      const uint32_t db = has_q ? (uint32_t)len * sizeof(TD) : 0u;
      mbar_expect_tx(&sm.bar, tb + db);
      if (tb) bulk_g2s(tbuf, trow + s0, tb, &sm.bar);
      if (db) bulk_g2s(dbuf, drow + s0, db, &sm.bar);
    }
  } else {
    for (int i = tid; i < len; i += kThreads) {
      tbuf[i] = trow[s0 + i];
      if (has_q) dbuf[i] = drow[s0 + i];
    }
  }
  // padding past the row end: target -inf; draft -inf logits or 0 probability
  for (int i = len + tid; i < slice; i += kThreads) {
    if constexpr (sizeof(TT) == 2) tbuf[i] = (TT)0xff80u;
    else reinterpret_cast<float*>(tbuf)[i] = neg_inf();
    if (has_q) {
      if constexpr (QK == Q_LOGITS) {
        if constexpr (sizeof(TD) == 2) dbuf[i] = (TD)0xff80u;
        else reinterpret_cast<float*>(dbuf)[i] = neg_inf();
      } else {
        dbuf[i] = (TD)0;
      }
    }
  }

  // ---- children of this row (warp 0)
  if (warp == 0) {
    int cnt = 0;
    uint32_t bad = 0;
    if (s.chain) {
      if (r < n) {
        if (lane == 0) {
          sm.kid_node[0] = r;
          sm.kid_tok[0] = a.node_tokens[(int64_t)b * n + r];
        }
        cnt = 1;
      }
    } else {
      const int32_t* par = a.parent + (int64_t)b * n;
      for (int j0 = 0; j0 < n; j0 += 32) {
        const int j = j0 + lane;
        int p = -2;
        if (j < n) p = par[j];
        const bool valid = (p >= -1 && p < j);
        if (j < n && !valid) bad |= SPEC_STATUS_BAD_TREE;
        const uint32_t m = __ballot_sync(0xffffffffu, j < n && valid && p == r - 1);
        if (m & (1u << lane)) {
          const int pos = cnt + __popc(m & ((1u << lane) - 1));
          if (pos < SPEC_MAX_CHILDREN) {
            sm.kid_node[pos] = j;
            sm.kid_tok[pos] = a.node_tokens[(int64_t)b * n + j];
          } else {
            bad |= SPEC_STATUS_BAD_TREE;
          }
        }
        cnt += __popc(m);
      }
      cnt = min(cnt, SPEC_MAX_CHILDREN);
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cnt > 0 && !has_q) {
        bad |= SPEC_STATUS_BAD_TREE;
        cnt = 0;
      }
      sm.nkids = cnt;
      if (rank == 0) flag_status(a.status, bad);
    }
  }
  if (P.bulk) {
    if (!mbar_wait_bounded(&sm.bar, 0)) flag_status(a.status, SPEC_STATUS_TIMEOUT);
  }
  __syncthreads();

  const int ntile = slice / kTile;
  const int tpw = ntile / kNW;
  const int tbeg = warp * tpw, tend = tbeg + tpw;

  // ---- pass A: online max / sum-exp per lane (base-2 domain)
  MaxSum mp{neg_inf(), 0.f}, mq{neg_inf(), 0.f};
  float zq_plain = 0.f;
  for (int t = tbeg; t < tend; ++t) {
    const int e = t * kTile + lane * 4;
    float v[4];
    ElemIO<TT>::get4(tbuf + e, v);
    float sv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sv[k] = __fmul_rn(v[k], P.kt);
    const float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    if (mt > mp.m) {
      mp.z *= ex2(mp.m - mt);
      mp.m = mt;
    }
    if (mp.m != neg_inf())
      mp.z += (ex2(sv[0] - mp.m) + ex2(sv[1] - mp.m)) + (ex2(sv[2] - mp.m) + ex2(sv[3] - mp.m));
    if (has_q) {
      float w[4];
      ElemIO<TD>::get4(dbuf + e, w);
      if constexpr (QK == Q_PROBS_T1) {
        zq_plain += (w[0] + w[1]) + (w[2] + w[3]);
      } else {
        float sq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          sq[k] = (QK == Q_LOGITS) ? __fmul_rn(w[k], P.kt) : __fmul_rn(lg2(w[k]), P.invT);
        const float m2 = fmaxf(fmaxf(sq[0], sq[1]), fmaxf(sq[2], sq[3]));
        if (m2 > mq.m) {
          mq.z *= ex2(mq.m - m2);
          mq.m = m2;
        }
        if (mq.m != neg_inf())
          mq.z += (ex2(sq[0] - mq.m) + ex2(sq[1] - mq.m)) + (ex2(sq[2] - mq.m) + ex2(sq[3] - mq.m));
      }
    }
  }
  mp = warp_ms(mp);
  if (QK == Q_PROBS_T1) zq_plain = warp_sum(zq_plain);
  else mq = warp_ms(mq);
  if (lane == 0) {
    sm.red[warp][0] = mp.m;
    sm.red[warp][1] = mp.z;
    sm.red[warp][2] = (QK == Q_PROBS_T1) ? 0.f : mq.m;
    sm.red[warp][3] = (QK == Q_PROBS_T1) ? zq_plain : mq.z;
  }
  __syncthreads();
  if (tid == 0) {
    MaxSum A{sm.red[0][0], sm.red[0][1]}, Bq{sm.red[0][2], sm.red[0][3]};
    float zq = sm.red[0][3];
    for (int k = 1; k < kNW; ++k) {
      A = ms_combine(A, MaxSum{sm.red[k][0], sm.red[k][1]});
      if (QK == Q_PROBS_T1) zq += sm.red[k][3];
      else Bq = ms_combine(Bq, MaxSum{sm.red[k][2], sm.red[k][3]});
    }
    sm.x[0].v[0] = A.m;
    sm.x[0].v[1] = A.z;
    sm.x[0].v[2] = (QK == Q_PROBS_T1) ? 0.f : Bq.m;
    sm.x[0].v[3] = (QK == Q_PROBS_T1) ? zq : Bq.z;
  }
  cluster_sync();
  if (tid == 0) {
    MaxSum A{neg_inf(), 0.f}, Bq{neg_inf(), 0.f};
    float zq = 0.f;
    for (int k = 0; k < C; ++k) {
      const uint32_t base = mapa(smem_u32(&sm.x[0].v[0]), (uint32_t)k);
      const MaxSum pa{ld_dsmem_f32(base), ld_dsmem_f32(base + 4)};
      A = ms_combine(A, pa);
      if (QK == Q_PROBS_T1) {
        zq += ld_dsmem_f32(base + 12);
      } else {
        const MaxSum pb{ld_dsmem_f32(base + 8), ld_dsmem_f32(base + 12)};
        Bq = ms_combine(Bq, pb);
      }
    }
    uint32_t bad = 0;
    if (!(A.z > 0.f) || !(A.m > neg_inf()) || isnan(A.z)) bad |= SPEC_STATUS_NAN;
    sm.Lp = A.m + log2f(A.z);
    if (has_q) {
      if (QK == Q_PROBS_T1) {
        if (!(zq > 0.f) || isnan(zq)) bad |= SPEC_STATUS_NAN;
        sm.invZq = 1.f / zq;
        sm.Lq = 0.f;
      } else {
        if (!(Bq.z > 0.f) || !(Bq.m > neg_inf()) || isnan(Bq.z)) bad |= SPEC_STATUS_NAN;
        sm.Lq = Bq.m + log2f(Bq.z);
        sm.invZq = 0.f;
      }
    } else {
      sm.Lq = 0.f;
      sm.invZq = 0.f;
    }
    if (rank == 0) flag_status(a.status, bad);
  }
  __syncthreads();

  Row<TT, TD, QK> row{tbuf, dbuf, P.kt, P.invT, -sm.Lp, -sm.Lq, sm.invZq};
  const int nk = sm.nkids;

  // point values at the children's tokens (read from global memory)
  if (warp == 0) {
    for (int k = lane; k < nk; k += 32) {
      const int x = sm.kid_tok[k];
      float pv = 0.f, qv = 0.f;
      if (x >= 0 && x < V) {
        pv = row.p_of(ElemIO<TT>::get(trow, x));
        qv = row.q_of(ElemIO<TD>::get(drow, x));
      }
      sm.kid_p[k] = pv;
      sm.kid_q[k] = qv;
    }
  }

  // ---- pass B: alpha, residual max(0, p - q), and p, per warp
  float acc_a = 0.f, acc_r = 0.f, acc_p = 0.f;
  for (int t = tbeg; t < tend; ++t) {
    const int e = t * kTile + lane * 4;
    float v[4];
    ElemIO<TT>::get4(tbuf + e, v);
    if (has_q) {
      float w[4];
      ElemIO<TD>::get4(dbuf + e, w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float p = row.p_of(v[k]);
        const float q = row.q_of(w[k]);
        const float mn = fminf(p, q);
        acc_a += mn;
        acc_r += p - mn;
        acc_p += p;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc_p += row.p_of(v[k]);
    }
  }
  acc_a = warp_sum(acc_a);
  acc_r = warp_sum(acc_r);
  acc_p = warp_sum(acc_p);
  if (lane == 0) {
    sm.wp[warp] = acc_p;
    sm.wr[warp] = acc_r;
    sm.red[warp][0] = acc_a;
  }
  __syncthreads();
  if (tid == 0) {
    float A = 0.f, Rr = 0.f, Pp = 0.f;
    for (int k = 0; k < kNW; ++k) {
      A += sm.red[k][0];
      Rr += sm.wr[k];
      Pp += sm.wp[k];
    }
    sm.x[1].v[0] = A;
    sm.x[1].v[1] = Rr;
    sm.x[1].v[2] = Pp;
  }
  cluster_sync();
  float alpha = 0.f, Rtot = 0.f, Ptot = 0.f;
  if (tid == 0) {
    alpha = gather_ranks(sm, 1, 0, C, nullptr);
    Rtot = gather_ranks(sm, 1, 1, C, sm.rk_r);
    Ptot = gather_ranks(sm, 1, 2, C, sm.rk_p);
    if (rank == 0) {
      if (s.chain) {
        if (r < n) a.mass[(int64_t)b * n + r] = alpha;
      } else {
        a.mass[unit] = has_q ? alpha : __int_as_float(0x7fc00000);
      }
    }
  }

  // ---- sibling recursion (cluster-uniform control flow)
  // Weight sources for the final draw: 0 = p (wp / rk_p), 1 = max(0, p - q)
  // (wr / rk_r), 2 + i = result of a sibling pass in buffer i (wx[i] / rkx[i]).
  float Cc = 0.f, W = 1.f, D = 1.f;   // residual constant, its mass, q mass left
  int accepted = -1;
  int src = 0, xb = 0, slot = 2;
  uint32_t st_bits = 0;
  for (int k = 0; k < nk; ++k) {
    if (tid == 0) {
      const int x = sm.kid_tok[k];
      int dec = 0;
      if (x < 0 || x >= V) {
        st_bits |= SPEC_STATUS_TOKEN_RANGE;
      } else {
        bool removed = false;
        for (int i = 0; i < k; ++i) removed |= (sm.kid_tok[i] == x);
        const float ax = resid_w(sm.kid_p[k], sm.kid_q[k], Cc);
        const float qj = removed ? 0.f : sm.kid_q[k] / D;
        if (qj == 0.f) {
          dec = 1;
          st_bits |= SPEC_STATUS_QZERO_ACCEPT;
        } else {
          const float u = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b,
                                         (uint32_t)sm.kid_node[k], 0u);
          dec = (u < (ax / W) / qj) ? 1 : 0;
        }
      }
      sm.decision = dec;
      sm.bc[0] = Cc + W / D;  // residual constant after this rejection
    }
    __syncthreads();
    if (sm.decision) {
      accepted = sm.kid_node[k];
      break;
    }
    const float Cn = sm.bc[0];
    float Wn = 0.f;
    int nsrc;
    if (Cc == 0.f && Cn == 1.f) {
      // max(0, p - q) was already summed in pass B
      if (tid == 0) Wn = Rtot;
      nsrc = 1;
    } else {
      float acc = 0.f;
      for (int t = tbeg; t < tend; ++t) {
        const int e = t * kTile + lane * 4;
        float v[4], w[4];
        ElemIO<TT>::get4(tbuf + e, v);
        ElemIO<TD>::get4(dbuf + e, w);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc += resid_w(row.p_of(v[j]), row.q_of(w[j]), Cn);
      }
      acc = warp_sum(acc);
      if (lane == 0) sm.wx[xb][warp] = acc;
      __syncthreads();
      if (tid == 0) {
        float tot = 0.f;
        for (int i = 0; i < kNW; ++i) tot += sm.wx[xb][i];
        sm.x[slot].v[0] = tot;
      }
      cluster_sync();
      if (tid == 0) Wn = gather_ranks(sm, slot, 0, C, sm.rkx[xb]);
      slot ^= 1;
      nsrc = 2 + xb;
    }
    if (tid == 0) {
      int upd = 0;
      if (Wn > 0.f) {
        Cc = Cn;
        W = Wn;
        upd = 1;
      } else {
        st_bits |= SPEC_STATUS_RESIDUAL_ZERO;  // keep p' as it was
      }
      const int x = sm.kid_tok[k];
      bool removed = false;
      for (int i = 0; i < k; ++i) removed |= (sm.kid_tok[i] == x);
      if (x >= 0 && x < V && !removed) D -= sm.kid_q[k];
      if (D <= 0.f) st_bits |= SPEC_STATUS_DRAFT_EXHAUSTED;
      sm.bc[1] = Cc;
      sm.bc[2] = (D <= 0.f) ? 1.f : 0.f;
      sm.bc[3] = (float)upd;
    }
    __syncthreads();
    Cc = sm.bc[1];
    if (sm.bc[3] != 0.f) {
      src = nsrc;
      if (nsrc >= 2) xb ^= 1;
    }
    const bool exhausted = sm.bc[2] != 0.f;
    __syncthreads();  // bc is rewritten by the next iteration
    if (exhausted) break;
  }

  // ---- draw from p' when no child was accepted
  if (accepted < 0) {
    // weights: p (Cc == 0) or max(0, p - Cc q); their per-warp and per-rank
    // totals come from the pass that produced them
    const float* wt = src == 0 ? sm.wp : (src == 1 ? sm.wr : sm.wx[src - 2]);
    if (tid == 0) {
      const float* rk = src == 0 ? sm.rk_p : (src == 1 ? sm.rk_r : sm.rkx[src - 2]);
      float tot = 0.f;
      for (int i = 0; i < C; ++i) tot += rk[i];
      const float u = philox_uniform(a.prm.seed, a.prm.philox_offset, (uint32_t)b, (uint32_t)r, 1u);
      float t = u * tot;
      int sel = -1;
      float pre = 0.f;
      for (int i = 0; i < C; ++i) {
        if (rk[i] > 0.f && pre + rk[i] > t) {
          sel = i;
          break;
        }
        pre += rk[i];
      }
      if (sel < 0) {  // rounding: last rank with mass, no crossing inside
        for (int i = C - 1; i >= 0; --i)
          if (rk[i] > 0.f) {
            sel = i;
            break;
          }
        pre = 0.f;
        for (int i = 0; i < sel; ++i) pre += rk[i];
        t = 3.0e38f;
      }
      sm.rank_sel = sel;
      sm.red[1][0] = t - pre;  // remaining threshold inside the selected rank
      sm.red[1][1] = -1.f;
      if (sel < 0) st_bits |= SPEC_STATUS_CDF_FALLBACK;
      // warp selection inside this CTA (meaningful only on rank `sel`)
      int wsel = -1;
      float wpre = 0.f;
      const float tt = t - pre;
      for (int i = 0; i < kNW; ++i) {
        if (wt[i] > 0.f && wpre + wt[i] > tt) {
          wsel = i;
          break;
        }
        wpre += wt[i];
      }
      if (wsel < 0) {
        for (int i = kNW - 1; i >= 0; --i)
          if (wt[i] > 0.f) {
            wsel = i;
            break;
          }
        wpre = 0.f;
        for (int i = 0; i < wsel; ++i) wpre += wt[i];
      }
      sm.red[1][2] = (float)wsel;
      sm.red[1][3] = tt - wpre;
    }
    __syncthreads();
    const int sel = sm.rank_sel;
    const int wsel = (int)sm.red[1][2];
    if (sel == (int)rank && warp == wsel && wsel >= 0) {
      const float thr = sm.red[1][3];
      float run = 0.f;
      int found = -1, lastpos = -1;
      for (int t = tbeg; t < tend && found < 0; ++t) {
        const int e = t * kTile + lane * 4;
        float v[4], w[4] = {0.f, 0.f, 0.f, 0.f};
        ElemIO<TT>::get4(tbuf + e, v);
        if (has_q && Cc != 0.f) ElemIO<TD>::get4(dbuf + e, w);
        float wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = (Cc == 0.f) ? row.p_of(v[j]) : resid_w(row.p_of(v[j]), row.q_of(w[j]), Cc);
        const float ls = (wv[0] + wv[1]) + (wv[2] + wv[3]);
        // inclusive scan of lane sums
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
            for (int j = 3; j >= 0; --j)
              if (wv[j] > 0.f) {
                lp = e + j;
                break;
              }
          }
          lp = __shfl_sync(0xffffffffu, lp, hl);
          lastpos = lp;
        }
        if (cross) {
          const int fl = __ffs(cross) - 1;
          int tok = -1;
          if (lane == fl) {
            float c = run + inc - ls;
            int last = -1;
            for (int j = 0; j < 4; ++j) {
              if (wv[j] > 0.f) last = e + j;
              c += wv[j];
              if (wv[j] > 0.f && c > thr) {
                tok = e + j;
                break;
              }
            }
            if (tok < 0) tok = last;  // rounding inside the lane
          }
          found = __shfl_sync(0xffffffffu, tok, fl);
        }
        run += __shfl_sync(0xffffffffu, inc, 31);
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
    if (sel < 0 && rank == 0 && tid == 0) a.row_token[unit] = 0;
  }
  if (rank == 0 && tid == 0) {
    a.row_child[unit] = accepted;
    if (st_bits) flag_status(a.status, st_bits);
  }
  cluster_sync();  // peers may still read this CTA's exchange slots
}

// Walk every sequence from its root along accepted children.
__global__ void sampled_walk(VerifyShape s, VerifyArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= s.B) return;
  const int n = s.n;
  const int64_t row0 = (int64_t)b * (n + 1);
  int32_t* out = a.out_tokens + row0;
  int r = 0, len = 0;
  while (true) {
    const int j = a.row_child[row0 + r];
    if (j < 0 || j >= n || len >= n) break;
    if (!s.chain) a.path_nodes[(int64_t)b * n + len] = j;
    out[len] = a.node_tokens[(int64_t)b * n + j];
    ++len;
    r = j + 1;
  }
  out[len] = a.row_token[row0 + r];
  for (int k = len + 1; k <= n; ++k) out[k] = -1;
  if (!s.chain)
    for (int k = len; k < n; ++k) a.path_nodes[(int64_t)b * n + k] = -1;
  a.count[b] = len;
}

template <typename TT, typename TD, int QK>
cudaError_t launch_units(const UnitParams& P, int C, cudaStream_t st) {
  const size_t dyn = (size_t)P.slice * (sizeof(TT) + sizeof(TD));
  auto kern = unit_full<TT, TD, QK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P.s.rows() * C));
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
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

// Cluster size and slice for a row of V logits: the smallest cluster whose
// per-CTA slices fit the shared-memory budget.
bool full_geometry(int V, int bytes_per_elem, int* C, int* slice) {
  const int budget = 200 * 1024;  // dynamic shared memory of one CTA
  for (int c = 1; c <= kMaxCluster; c *= 2) {
    const int sl = ((V + c - 1) / c + kSliceQuant - 1) / kSliceQuant * kSliceQuant;
    if ((int64_t)sl * bytes_per_elem <= budget) {
      *C = c;
      *slice = sl;
      return true;
    }
  }
  return false;
}

// Full-vocabulary sampled verification can run: the streaming kernel takes
// 16-byte aligned rows, the general kernel any row whose slice fits one
// CTA's shared memory in a cluster of up to 8.
bool sampled_supported(const VerifyShape& s, const VerifyArgs& a) {
  if (truncation_k(&a.prm, s.V) > 0) return true;
  const int tsz = a.dt_target == SPEC_BF16 ? 2 : 4;
  const int dsz = a.dt_draft == SPEC_BF16 ? 2 : 4;
  const bool al_t = ((uintptr_t)a.target % 16 == 0) && ((int64_t)s.V * tsz % 16 == 0);
  const bool al_d = (a.draft == nullptr) || (((uintptr_t)a.draft % 16 == 0) && ((int64_t)s.V * dsz % 16 == 0));
  int c, sl, nch, ns;
  if (al_t && al_d && stream_geometry(s.V, tsz, dsz, &c, &sl, &nch, &ns)) return true;
  return full_geometry(s.V, tsz + dsz, &c, &sl);
}

cudaError_t launch_sampled(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st) {
  if (s.B == 0) return cudaSuccess;
  const int tk = truncation_k(&a.prm, s.V);
  if (tk > 0) {
    if (!a.topk_idx || !a.topk_val || !a.topk_cnt || !a.meta) return cudaErrorInvalidValue;
    return launch_sparse(s, a, tk, st);
  }
  UnitParams P{};
  P.s = s;
  P.a = a;
  const int tsz = a.dt_target == SPEC_BF16 ? 2 : 4;
  const int dsz = a.dt_draft == SPEC_BF16 ? 2 : 4;
  int C = 1, slice = 0;
  const bool full_ok = full_geometry(s.V, tsz + dsz, &C, &slice);
  P.slice = slice;
  const bool al_t = ((uintptr_t)a.target % 16 == 0) && ((int64_t)s.V * tsz % 16 == 0);
  const bool al_d = (a.draft == nullptr) || (((uintptr_t)a.draft % 16 == 0) && ((int64_t)s.V * dsz % 16 == 0));
  P.bulk = (al_t && al_d) ? 1 : 0;
  const float T = a.prm.temperature;
  P.kt = kLog2e / T;
  P.invT = 1.f / T;
  const int qk = a.prm.draft_kind == SPEC_DRAFT_LOGITS ? Q_LOGITS : (T == 1.f ? Q_PROBS_T1 : Q_PROBS_T);
  cudaError_t e = cudaSuccess;
  // bandwidth path: persistent streaming clusters (16-byte aligned rows)
  StreamParams Q{};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // a few sampled chains: one launch, every row resident in shared memory
  int cs_slice = 0;
  size_t cs_smem = 0;
  if (!a.tlse && chain_small_fits(s, a, sms, &cs_slice, &cs_smem))
    return launch_chain_small(s, a, cs_slice, cs_smem, st);
  // pass A reads the target row unless its normaliser is given (LM head
  // epilogue), and the draft row unless its normaliser is given
  const int passA = (a.tlse ? 0 : tsz) + ((qk == Q_LOGITS && a.prm.draft_lse) ? 0 : dsz);
  if (P.bulk && a.meta && a.qres && a.rowout &&
      stream_geometry(s.V, tsz, dsz, &Q.C, &Q.slice, &Q.nch, &Q.stages, s.rows(), sms,
                      passA)) {
    Q.s = s;
    Q.a = a;
    Q.qk = qk;
    Q.kt = P.kt;
    Q.invT = P.invT;
    Q.kidcap = meta_kidcap(s.chain);
    Q.rec_bytes = meta_rec_bytes(s.chain);
    return (a.dt_target == SPEC_BF16) ? launch_stream_bf16(Q, st) : launch_stream_f32(Q, st);
  }
  if (!full_ok) return cudaErrorNotSupported;
  prof_begin(SPEC_PROF_VERIFY, st);
#define SV_DISPATCH(TT, TD)                                     \
  if (qk == Q_LOGITS) e = launch_units<TT, TD, Q_LOGITS>(P, C, st); \
  else if (qk == Q_PROBS_T1) e = launch_units<TT, TD, Q_PROBS_T1>(P, C, st); \
  else e = launch_units<TT, TD, Q_PROBS_T>(P, C, st);
  if (a.dt_target == SPEC_BF16) {
    if (a.dt_draft == SPEC_BF16) { SV_DISPATCH(uint16_t, uint16_t) }
    else { SV_DISPATCH(uint16_t, float) }
  } else {
    if (a.dt_draft == SPEC_BF16) { SV_DISPATCH(float, uint16_t) }
    else { SV_DISPATCH(float, float) }
  }
#undef SV_DISPATCH
  prof_end(SPEC_PROF_VERIFY, st);
  if (e != cudaSuccess) return e;
  sampled_walk<<<(s.B + 127) / 128, 128, 0, st>>>(s, a);
  return cudaGetLastError();
}

}  // namespace sv
