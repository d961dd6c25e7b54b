// Streaming sampled verification (temperature > 0, full vocabulary): the
// bandwidth path for rows whose logits are 16-byte aligned.
//
// The method ("064 · 投机解码", sections 二-三; EAGLE-2 notes §2.1-2.2): p and
// q are the softmaxes of the transformed target and draft rows; a drafted
// child with token x is accepted iff u < p'(x) / q'(x); siblings are tried
// in index order with the unrolled residual max(0, p - C q); a row whose
// children are all rejected (or a leaf) draws its token by inverse CDF in
// vocabulary order.
//
// GB300 organisation.  A row needs two passes over its logits: one for the
// softmax normalisers, one for alpha = sum min(p, q) and the residual mass.
// Holding a row on chip between them caps the rows in flight and leaves the
// kernel latency-bound, so instead:
//  * persistent clusters of C CTAs (C = 2: 76 clusters cover all 152 SMs);
//    CTA `rank` owns one contiguous vocabulary slice of every row of its
//    cluster; rows go round-robin over clusters;
//  * a producer warp streams 4096-logit chunks with TMA bulk copies into a
//    ring of shared-memory stages; each stage carries chunk c of row j (pass
//    A: online max / sum of p and q) AND chunk c of row j - 1 (pass B), so
//    pass B re-reads a row one row-time after pass A.  Pass A's copies are
//    marked evict_last and pass B's evict_first, so the second read hits L2
//    and HBM sees each byte once;
//  * at the end of each row-time the CTA's statistics of row j and residual
//    mass of row j - 1 travel to the peers in one 32-byte st.async per peer;
//    they are waited for at the start of the next row-time, so the cluster
//    exchange sits off the streaming path;
//  * decisions run one and two row-times behind: the first child's test
//    needs only the normalisers, the second child's only the residual mass
//    R of max(0, p - q); whatever needs the mass of max(0, p - C q) for a
//    new C (a third child, or the draw after the last rejection) is left to
//    the walk, which finishes the recursion only for the rows on the
//    accepted path, with one pass over the row per C.

#pragma once

#include <climits>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace stream {
namespace {  // internal to each translation unit that instantiates it

constexpr int kCW = 16;             // consumer warps
constexpr int kCT = kCW * 32;       // consumer threads
constexpr int kThreads = kCT + 64;  // + a producer warp and a control warp
constexpr int kEPT = 8;             // logits per consumer thread per chunk
constexpr int kCH = kCT * kEPT;     // logits per chunk (4096)
constexpr int kMaxC = 4;
constexpr int kMaxNS = 8;
constexpr int kRing = 192 * 1024;   // shared-memory ring bytes
constexpr int kMaxTiles = 32;       // chunks per slice the walk's draw handles
constexpr int kMaxKids = SPEC_MAX_CHILDREN;
constexpr int kBar = 1;             // named barrier of the consumer warps

enum QKind { Q_LOGITS = 0, Q_PROBS_T1 = 1, Q_PROBS_T = 2 };

// Per-row record built by row_meta.  Global layout (stride rec_bytes):
// header, kid[kidcap], then kidcap floats of accept uniforms; copied byte for
// byte to the start of a shared-memory Meta, so the uniforms of a record
// with kidcap slots start at &kid[kidcap].
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

// One warp per row: the row's draft row, its children in index order with
// their tokens and the two logits at each token, and its Philox uniforms
// (slot 0 of each child, slot 1 of the row), so that the streaming kernel
// issues no dependent loads and no Philox rounds.  With a.qlist set the row
// also goes on the streaming kernel's work list (or, without a draft row,
// gets its final row outcome).
template <typename TT, typename TD>
__device__ void row_meta_warp(const VerifyShape& s, const VerifyArgs& a, int64_t unit, int lane,
                              int kidcap, int rec_bytes) {
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
    if (a.qlist) {
      if (qr >= 0) {  // the streaming kernel's work: rows that have a draft row
        a.qlist[atomicAdd(a.qcount, 1)] = (int32_t)unit;
      } else {
        // a row without a draft row has no children and no acceptance mass;
        // the walk finds its normaliser only if it draws there (Lp = NaN)
        RowOut o{};
        o.child = -1;
        o.W = 1.f;
        o.D = 1.f;
        o.Lp = __int_as_float(0x7fc00000);
        o.bits = bad;
        a.rowout[unit] = o;
        flag_status(a.status, bad);
      }
    }
  }
}
template <typename TT, typename TD>
__global__ void __launch_bounds__(256) row_meta(VerifyShape s, VerifyArgs a, int kidcap,
                                                int rec_bytes) {
  launch_dependents();  // the streaming kernel waits for this grid itself
  const int64_t unit = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (unit >= s.rows()) return;
  row_meta_warp<TT, TD>(s, a, unit, threadIdx.x & 31, kidcap, rec_bytes);
}

// State of a row between its first decision and its last (two row-times).
struct RowState {
  float Lp, Lq, invZq;  // base-2 log normalisers (invZq: probabilities at T = 1)
  int accepted;         // accepted child node, -1 none yet
  int pending;          // 1: child 0 was rejected, the rest waits for R
  uint32_t bits;        // status bits so far
};

struct Smem {
  uint64_t full[kMaxNS], empty[kMaxNS];
  uint64_t mrec[3], recfree[3];
  uint64_t xbar[4];           // one stream exchange per row-time (ring of 4)
  float4 xslot[4][kMaxC][2];  // [row-time][rank]{stats of row j, residual of row j-1}
  Meta rec[3];
  float4 wst[2][kCW];         // per-warp statistics (double-buffered by row-time)
  float2 wab[2][kCW];         // per-warp alpha / residual
  RowState rs[2];
  uint64_t dec[2];            // control warp -> consumers: needR of the pass-B row
  int needR[2];
  int dead;                   // a bounded wait gave up: skip the remaining waits
};

__device__ __forceinline__ float resid_w(float p, float q, float C) {
  return C == 0.f ? p : fmaxf(0.f, fmaf(-C, q, p));
}

// Waits that give up after ~1 s, flag SPEC_STATUS_TIMEOUT and make every
// later wait of the CTA return at once, so a broken peer cannot hang the GPU.
// A phase that is already complete returns after one test, before the flag
// (a shared-memory load) is read.
__device__ __forceinline__ void wait_cta(Smem& sm, uint64_t* bar, uint32_t parity,
                                         uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return;
  if (*(volatile int*)&sm.dead) return;
  if (!mbar_wait_bounded(bar, parity)) {
    sm.dead = 1;
    flag_status(status, SPEC_STATUS_TIMEOUT);
  }
}
__device__ __forceinline__ void wait_cluster(Smem& sm, uint64_t* bar, uint32_t parity,
                                             uint32_t* status) {
  if (mbar_try_wait_cluster(bar, parity)) return;
  if (*(volatile int*)&sm.dead) return;
  if (!mbar_wait_cluster_bounded(bar, parity)) {
    sm.dead = 1;
    flag_status(status, SPEC_STATUS_TIMEOUT);
  }
}

__device__ __forceinline__ void bulk_g2s_pol(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Eight consecutive elements from 16-byte aligned memory, widened to float.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float v[8]);
template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, float v[8]) {
  const uint4 x = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
  v[4] = bf16_lo(x.z); v[5] = bf16_hi(x.z); v[6] = bf16_lo(x.w); v[7] = bf16_hi(x.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float v[8]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  const float4 y = *reinterpret_cast<const float4*>(p + 4);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}
// The same from global memory without L1 allocation (continuation passes and
// the walk's draw).
template <typename T>
__device__ __forceinline__ void ldg8(const T* p, float v[8]);
template <>
__device__ __forceinline__ void ldg8<uint16_t>(const uint16_t* p, float v[8]) {
  uint4 x;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "l"(p));
  v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
  v[4] = bf16_lo(x.z); v[5] = bf16_hi(x.z); v[6] = bf16_lo(x.w); v[7] = bf16_hi(x.w);
}
template <>
__device__ __forceinline__ void ldg8<float>(const float* p, float v[8]) {
  float4 x, y;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
               : "l"(p));
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(y.x), "=f"(y.y), "=f"(y.z), "=f"(y.w)
               : "l"(p + 4));
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

// Raw 16-byte loads of 8 elements (no conversion), so that several chunks
// can be in flight before any is used; unpack8 widens them afterwards.
template <typename T>
struct Raw8 {
  uint4 w[sizeof(T) / 2];
};
template <typename T>
__device__ __forceinline__ void ldg_raw(const T* p, Raw8<T>& r) {
#pragma unroll
  for (int i = 0; i < (int)(sizeof(T) / 2); ++i)
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.w[i].x), "=r"(r.w[i].y), "=r"(r.w[i].z), "=r"(r.w[i].w)
                 : "l"(reinterpret_cast<const unsigned char*>(p) + 16 * i));
}
__device__ __forceinline__ void unpack8(const Raw8<uint16_t>& r, float v[8]) {
  const uint4 x = r.w[0];
  v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
  v[4] = bf16_lo(x.z); v[5] = bf16_hi(x.z); v[6] = bf16_lo(x.w); v[7] = bf16_hi(x.w);
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float v[8]) {
  v[0] = __uint_as_float(r.w[0].x); v[1] = __uint_as_float(r.w[0].y);
  v[2] = __uint_as_float(r.w[0].z); v[3] = __uint_as_float(r.w[0].w);
  v[4] = __uint_as_float(r.w[1].x); v[5] = __uint_as_float(r.w[1].y);
  v[6] = __uint_as_float(r.w[1].z); v[7] = __uint_as_float(r.w[1].w);
}
// Chunks of plain loads in flight per thread: eight 16-byte registers' worth.
template <typename TT, typename TD>
constexpr int inflight() {
  return 16 / (int)(sizeof(TT) + sizeof(TD)) > 0 ? 16 / (int)(sizeof(TT) + sizeof(TD)) : 1;
}

// q at one element of a draft row, given the row's normalisers.
template <int QK>
__device__ __forceinline__ float q_of(float raw, float kt, float invT, float negLq, float invZq) {
  if constexpr (QK == Q_LOGITS) return ex2(fmaf(raw, kt, negLq));
  else if constexpr (QK == Q_PROBS_T1) return __fmul_rn(raw, invZq);
  else return ex2(fmaf(lg2(raw), invT, negLq));
}

__device__ __forceinline__ float2 ex2x2(float2 t) { return make_float2(ex2(t.x), ex2(t.y)); }

// Online sum of 2^(x_i s - m) over a thread's logits with a lazy reference m:
// the exponentials use the current m, which moves up (rescaling the sum) only
// when a group's sum would pass 2^60, so the common path has no dependency on
// the group's maximum; z stays below 2^64 per 16 groups, far from overflow.
// (m, z) then combine like a (max, sum) pair; m = -inf until a finite logit.
__device__ __forceinline__ void lazy_sum(const float (&x)[8], float s, float& m, float& z) {
  float2 zc2 = make_float2(0.f, 0.f);
  {
    const float2 s2 = make_float2(s, s), nm2 = make_float2(-m, -m);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      zc2 = fadd2(zc2, ex2x2(ffma2(make_float2(x[i], x[i + 1]), s2, nm2)));
  }
  float zc = zc2.x + zc2.y;
  if (!(zc <= 0x1p60f)) {  // a new maximum (or the first finite logit, or NaN)
    const float cm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                           fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
    const float mn = fmaxf(m, __fmul_rn(cm, s));
    zc = 0.f;
    if (mn != neg_inf()) {
      if (m != neg_inf()) z *= ex2(m - mn);
      m = mn;
#pragma unroll
      for (int i = 0; i < 8; ++i) zc += ex2(fmaf(x[i], s, -m));
    }
  }
  z += zc;
}

// Test of child k of a row (u = its accept uniform): accepted iff
// u < (r(x) / W) / (q(x) / D) with r = max(0, p - Cc q) (p when Cc = 0), W its
// mass and D the draft mass left after the rejected siblings; a token already
// rejected has q' = 0 and a token with q'(x) = 0 is accepted (flagged).
template <int QK>
__device__ __forceinline__ int child_test(const Meta& M, int kidcap, int k, float Cc, float W,
                                          float D, const RowState& S, float kt, float invT,
                                          int V, uint32_t* bits) {
  const int x = M.kid[k].tok;
  if (x < 0 || x >= V) {
    *bits |= SPEC_STATUS_TOKEN_RANGE;
    return 0;
  }
  bool removed = false;
  for (int i = 0; i < k; ++i) removed |= (M.kid[i].tok == x);
  const float pv = ex2(fmaf(M.kid[k].raw_t, kt, -S.Lp));
  const float qv = q_of<QK>(M.kid[k].raw_q, kt, invT, -S.Lq, S.invZq);
  const float ax = resid_w(pv, qv, Cc);
  const float qj = removed ? 0.f : qv / D;
  if (qj == 0.f) {
    *bits |= SPEC_STATUS_QZERO_ACCEPT;
    return 1;
  }
  const float* uk = reinterpret_cast<const float*>(&M.kid[kidcap]);
  return (uk[k] < (ax / W) / qj) ? 1 : 0;
}

// The sibling recursion of a row from the state "child st.k was rejected,
// the next residual coefficient is st.Cn" (st.D already reduced by that
// child's q when `reduced`).  Wn is the mass of max(0, p - st.Cn q) if known
// (< 0 otherwise), R the mass of max(0, p - q) if known (< 0 otherwise).
// On return st.child is the accepted child, -1 (the row ends: its token is
// drawn from max(0, p - Cn q), or max(0, p - Cc q) if that has no mass) or
// -2 (the next step needs the mass for st.Cn: one more pass).  This is the
// unrolled form of p' <- norm(max(0, p' - q')), q' <- q' without the rejected
// token, with the order of the original: residual, remove, stop if the draft
// mass is gone or no child is left, test the next child.
template <int QK>
__device__ void siblings(const Meta& M, int kidcap, RowOut& st, float Wn, float R, bool reduced,
                         float kt, float invT, int V) {
  const RowState S{st.Lp, st.Lq, st.invZq, -1, 0, 0u};
  for (;;) {
    if (!reduced) {
      const int x = M.kid[st.k].tok;
      bool removed = false;
      for (int i = 0; i < st.k; ++i) removed |= (M.kid[i].tok == x);
      if (x >= 0 && x < V && !removed) st.D -= q_of<QK>(M.kid[st.k].raw_q, kt, invT, -st.Lq, st.invZq);
      if (st.D <= 0.f) {
        st.bits |= SPEC_STATUS_DRAFT_EXHAUSTED;
        st.child = -1;
        return;
      }
      if (st.k + 1 >= M.nk) {
        st.child = -1;
        return;
      }
      reduced = true;
    }
    if (Wn < 0.f) {
      if (R >= 0.f && st.Cc == 0.f && st.Cn == 1.f) {
        Wn = R;
      } else {
        st.child = -2;
        return;
      }
    }
    if (Wn > 0.f) {
      st.Cc = st.Cn;
      st.W = Wn;
    } else {
      st.bits |= SPEC_STATUS_RESIDUAL_ZERO;
    }
    ++st.k;
    if (child_test<QK>(M, kidcap, st.k, st.Cc, st.W, st.D, S, kt, invT, V, &st.bits)) {
      st.child = M.kid[st.k].node;
      return;
    }
    st.Cn = st.Cc + st.W / st.D;
    Wn = -1.f;
    reduced = false;
  }
}

template <typename TT, typename TD, int QK>
__global__ void __launch_bounds__(kThreads, 1) unit_stream(StreamParams P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  // a programmatic dependent of row_meta (records, row list and count): it
  // reads nothing before that grid has completed; the walk may then be
  // scheduled as this grid's CTAs leave
  grid_dependency_wait();
  launch_dependents();
  const VerifyShape& s = P.s;
  const VerifyArgs& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int C = P.C;
  const int cid = blockIdx.x / C;
  const int ncl = P.nclusters;
  const int64_t nunits = *reinterpret_cast<volatile const int32_t*>(a.qcount);  // rows with a draft row
  // when every row has a draft row the list is all rows: keep row order
  const bool ident = nunits == s.rows();
  auto unit_of = [&](int j) -> int64_t {
    const int64_t i = cid + (int64_t)j * ncl;
    return ident ? i : (int64_t)a.qlist[i];
  };
  const int V = s.V, n = s.n;
  const int r0 = (int)rank * P.slice;
  const int len = max(0, min(P.slice, V - r0));
  const int nch = (len + kCH - 1) / kCH;
  const int nrow = (cid < nunits) ? (int)((nunits - cid + ncl - 1) / ncl) : 0;
  const int NS = P.stages;
  const float kt = P.kt, invT = P.invT;
  constexpr size_t kTB = (size_t)kCH * sizeof(TT);
  constexpr size_t kHalf = (size_t)kCH * (sizeof(TT) + sizeof(TD));
  auto stage = [&](int st, int half) { return dyn + (size_t)st * 2 * kHalf + half * kHalf; };
  const TT* tgt = reinterpret_cast<const TT*>(a.target);
  const TD* drf = reinterpret_cast<const TD*>(a.draft);
  // the caller's draft-row normalisers (logit drafts only): pass A then
  // reads the target row alone and the draft row is read once, in pass B
  const float* qlse = QK == Q_LOGITS ? a.prm.draft_lse : nullptr;
  // the target rows' normalisers, when the LM head's epilogue computed them:
  // pass A then leaves the target row out and pass B reads it once
  const float* plse = a.tlse;
  auto draft_row = [&](int64_t u, int q) -> const TD* {
    const int64_t b = u / (n + 1);
    return drf + ((int64_t)b * s.R + q) * V;
  };

  if (tid == 0) {
    sm.dead = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kCW);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sm.mrec[i], 1);
      mbar_init(&sm.recfree[i], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&sm.xbar[i], 1);
    for (int i = 0; i < 2; ++i) mbar_init(&sm.dec[i], 1);
    fence_mbar_init();
  }
  cluster_sync();  // every CTA's barriers exist before the first st.async

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nrow > 0) {
      uint64_t pol_a, pol_b;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_a));
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_b));
      int stg = 0, round = 0;
      // this cluster's rows: qlist[cid + j * ncl]; unit ids and draft rows
      // are read two and one rows ahead of their use
      int64_t u_cur = unit_of(0), u_prev = -1;
      int64_t u_nxt = (1 < nrow) ? unit_of(1) : -1;
      int q_cur = a.qres[u_cur], q_prev = -1;
      for (int j = 0; j <= nrow; ++j) {
        const bool hA = j < nrow, hB = j >= 1;
        const int64_t ua = u_cur, ub = u_prev;
        const int qa = hA ? q_cur : -1, qb = hB ? q_prev : -1;
        const int64_t u_nn = (j + 2 < nrow) ? unit_of(j + 2) : -1;
        const int q_next = (u_nxt >= 0) ? a.qres[u_nxt] : -1;
        if (hA) {  // row j's record: read at its first decision and its last
          const int rb = j % 3;
          if (j >= 3) wait_cta(sm, &sm.recfree[rb], (uint32_t)(((j / 3) - 1) & 1), a.status);
          mbar_expect_tx(&sm.mrec[rb], (uint32_t)P.rec_bytes);
          bulk_g2s(&sm.rec[rb], a.meta + ua * (int64_t)P.rec_bytes, (uint32_t)P.rec_bytes,
                   &sm.mrec[rb]);
        }
        const TT* ta = (hA && !plse) ? tgt + ua * (int64_t)V + r0 : nullptr;
        const TD* da = (qa >= 0 && !qlse) ? draft_row(ua, qa) + r0 : nullptr;
        const TT* tb = hB ? tgt + ub * (int64_t)V + r0 : nullptr;
        const TD* db = qb >= 0 ? draft_row(ub, qb) + r0 : nullptr;
        for (int c = 0; c < nch; ++c) {
          if (round > 0) wait_cta(sm, &sm.empty[stg], (uint32_t)((round - 1) & 1), a.status);
          const int v = min(kCH, len - c * kCH);
          const uint32_t bt = (uint32_t)v * sizeof(TT), bd = (uint32_t)v * sizeof(TD);
          uint32_t bytes = 0;
          if (ta) bytes += bt;
          if (da) bytes += bd;
          if (db) bytes += bt + bd;
          mbar_expect_tx(&sm.full[stg], bytes);
          unsigned char* sa = stage(stg, 0);
          unsigned char* sb = stage(stg, 1);
          if (ta) bulk_g2s_pol(sa, ta + c * kCH, bt, &sm.full[stg], pol_a);
          if (da) bulk_g2s_pol(sa + kTB, da + c * kCH, bd, &sm.full[stg], pol_a);
          if (db) {
            bulk_g2s_pol(sb, tb + c * kCH, bt, &sm.full[stg], pol_b);
            bulk_g2s_pol(sb + kTB, db + c * kCH, bd, &sm.full[stg], pol_b);
          }
          if (++stg == NS) {
            stg = 0;
            ++round;
          }
        }
        q_prev = qa;
        q_cur = q_next;
        u_prev = ua;
        u_cur = u_nxt;
        u_nxt = u_nn;
      }
    }
  } else {
    // ------------------------------------------- consumers and control warp
    const bool ctl = warp == kCW + 1;
    int stg = 0, round = 0;
    float Lp = 0.f, Lq = 0.f, invZq = 0.f;  // normalisers of the pass-B row
    float zp_tot = 0.f, zq_tot = 0.f;
    int64_t u_cur = nrow > 0 ? unit_of(0) : -1, u_prev = -1, u_prev2 = -1;
    int q_cur = nrow > 0 ? a.qres[u_cur] : -1, q_prev = -1;
    float lq_carry = 0.f, lp_carry = 0.f;
    for (int j = 0; nrow > 0 && j <= nrow + 1; ++j) {
      const bool hA = j < nrow, hB = j >= 1 && j <= nrow;
      const int qa = hA ? q_cur : -1, qb = hB ? q_prev : -1;
      const int64_t u_next = (j + 1 < nrow) ? unit_of(j + 1) : -1;
      const int q_next = (u_next >= 0) ? a.qres[u_next] : -1;
      const int64_t ub = u_prev, ur2 = u_prev2;
      const float lq_b = lq_carry;  // row j - 1's given normalisers
      const float lp_b = lp_carry;
      lq_carry = (qlse && qa >= 0) ? __ldg(qlse + (u_cur / (n + 1)) * s.R + qa) : 0.f;
      lp_carry = (plse && hA) ? __ldg(plse + u_cur) : 0.f;

      // Steps 1-3: the previous row-time's exchange and the decisions it allows.
      auto row_start = [&]() {
        // 1. statistics of row j - 1 (and residual mass of row j - 2)
        if (j >= 1) {
          const int xs = (j - 1) & 3;
          wait_cluster(sm, &sm.xbar[xs], (uint32_t)(((j - 1) >> 2) & 1), a.status);
          if (hB) {
            const float4 v = (lane < C) ? sm.xslot[xs][lane][0]
                                        : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
            MaxSum A{v.x, v.y}, Bq{v.z, v.w};
            float z1 = (lane < C) ? v.w : 0.f;
  #pragma unroll
            for (int o = kMaxC / 2; o > 0; o >>= 1) {
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
            Lp = A.m + log2f(A.z);
            zp_tot = A.z;
            if (plse) {  // given: finite unless the row is empty or not a number
              Lp = lp_b;
              zp_tot = (fabsf(lp_b) < 0x1p126f) ? 1.f : 0.f;
            }
            Lq = 0.f;
            invZq = 0.f;
            zq_tot = 0.f;
            if (qb >= 0) {
              if (QK == Q_PROBS_T1) {
                zq_tot = __shfl_sync(0xffffffffu, z1, 0);
                invZq = 1.f / zq_tot;
              } else {
                Bq.m = __shfl_sync(0xffffffffu, Bq.m, 0);
                Bq.z = __shfl_sync(0xffffffffu, Bq.z, 0);
                Lq = Bq.m + log2f(Bq.z);
                zq_tot = Bq.z;
                if (qlse) {  // given: finite unless the row is empty or not a number
                  Lq = lq_b;
                  zq_tot = (fabsf(lq_b) < 0x1p126f) ? 1.f : 0.f;
                }
              }
            }
          }
        }

        // 3. first decision of row j - 1 (needs only its normalisers; control)
        if (hB && ctl && lane == 0) {
          const int rb = (j - 1) % 3;
          wait_cta(sm, &sm.mrec[rb], (uint32_t)(((j - 1) / 3) & 1), a.status);
          const Meta& M = sm.rec[rb];
          const RowState S0{Lp, Lq, invZq, -1, 0, 0u};
          uint32_t bits = 0;
          int acc0 = -1;
          if (M.nk > 0 && child_test<QK>(M, P.kidcap, 0, 0.f, 1.f, 1.f, S0, kt, invT, V, &bits))
            acc0 = M.kid[0].node;
          if (rank == 0) {
            if (!(zp_tot > 0.f) || isnan(zp_tot)) bits |= SPEC_STATUS_NAN;
            if (qb >= 0 && (!(zq_tot > 0.f) || isnan(zq_tot))) bits |= SPEC_STATUS_NAN;
          }
          RowState& S = sm.rs[(j - 1) & 1];
          S.Lp = Lp;
          S.Lq = Lq;
          S.invZq = invZq;
          S.accepted = acc0;
          S.pending = (M.nk > 0 && acc0 < 0) ? 1 : 0;
          S.bits = bits;
          // pass B needs R only for a second child's test
          sm.needR[(j - 1) & 1] = (M.nk >= 2 && acc0 < 0) ? 1 : 0;
          mbar_arrive(&sm.dec[(j - 1) & 1]);
        }


        // 2. decisions of row j - 2 that need its residual mass R (control)
        if (j >= 2 && ctl && lane == 0) {
          const int rr = j - 2;
          const int64_t ur = ur2;
          const RowState& S = sm.rs[rr & 1];
          const Meta& M = sm.rec[rr % 3];
          RowOut st{};
          st.child = -1;
          st.k = 0;
          st.Cc = 0.f;
          st.W = 1.f;
          st.D = 1.f;
          st.Cn = 0.f;  // a leaf draws from p
          st.Lp = S.Lp;
          st.Lq = S.Lq;
          st.invZq = S.invZq;
          st.bits = S.bits | M.bad;
          if (S.accepted >= 0) {
            st.child = S.accepted;
          } else if (S.pending) {  // child 0 rejected: Cn = 1, whose mass is R
            const float4(*rx)[2] = sm.xslot[(rr + 1) & 3];
            float R = 0.f;
            for (int i = 0; i < C; ++i) R += rx[i][1].x;
            st.Cn = 1.f;
            siblings<QK>(M, P.kidcap, st, -1.f, R, false, kt, invT, V);
          }
          if (rank == 0) {
            a.rowout[ur] = st;
            flag_status(a.status, st.bits);
          }
          mbar_arrive(&sm.recfree[rr % 3]);
        }

      };

      // 4. one row-time of chunks: pass A of row j, pass B of row j - 1 (the
      // control warp only takes the decisions)
      row_start();
      if (j > nrow) break;
      if (ctl) {
        q_prev = qa;
        q_cur = q_next;
        u_prev2 = u_prev;
        u_prev = u_cur;
        u_cur = u_next;
        continue;
      }
      bool needR = false;
      if (qb >= 0) {
        wait_cta(sm, &sm.dec[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), a.status);
        needR = sm.needR[(j - 1) & 1] != 0;
      }
      float m = neg_inf(), z = 0.f, mq = neg_inf(), zq = 0.f;
      float2 acc_a2 = make_float2(0.f, 0.f), acc_r2 = make_float2(0.f, 0.f), zq2 = make_float2(0.f, 0.f);
      const float2 kt2 = make_float2(kt, kt);
      // The chunk loop, one instantiation per combination of the row-time's
      // uniform choices (whether pass A sums the target row and whether it
      // sums the draft row, pass B present and whether it needs the residual
      // mass), so that the loop body tests none of them.
      auto chunk_loop = [&](auto fA, auto fQ, auto fB, auto fR) {
        constexpr bool kA = decltype(fA)::value, kQ = decltype(fQ)::value;
        constexpr bool kB = decltype(fB)::value, kR = decltype(fR)::value;
        for (int c = 0; c < nch; ++c) {
          wait_cta(sm, &sm.full[stg], (uint32_t)(round & 1), a.status);
          const int e = c * kCH + tid * kEPT;
          if (e < len) {  // len is a multiple of 8: the thread's 8 logits are all valid
            if constexpr (kA) {
              const unsigned char* sa = stage(stg, 0);
              float x[8];
              load8<TT>(reinterpret_cast<const TT*>(sa) + tid * kEPT, x);
              lazy_sum(x, kt, m, z);
            }
            if constexpr (kQ) {
              const unsigned char* sa = stage(stg, 0);
              float y[8];
              load8<TD>(reinterpret_cast<const TD*>(sa + kTB) + tid * kEPT, y);
              if constexpr (QK == Q_PROBS_T1) {
                zq2 = fadd2(zq2, fadd2(fadd2(make_float2(y[0], y[1]), make_float2(y[2], y[3])),
                                       fadd2(make_float2(y[4], y[5]), make_float2(y[6], y[7]))));
              } else if constexpr (QK == Q_LOGITS) {
                lazy_sum(y, kt, mq, zq);
              } else {
  #pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = lg2(y[i]);
                lazy_sum(y, invT, mq, zq);
              }
            }
            if constexpr (kB) {
              const float negLp = -Lp, negLq = -Lq;
              const unsigned char* sb = stage(stg, 1);
              float x[8], y[8];
              load8<TT>(reinterpret_cast<const TT*>(sb) + tid * kEPT, x);
              load8<TD>(reinterpret_cast<const TD*>(sb + kTB) + tid * kEPT, y);
              const float2 nLp2 = make_float2(negLp, negLp), nLq2 = make_float2(negLq, negLq);
              auto q2_of = [&](int i) -> float2 {
                if constexpr (QK == Q_LOGITS)
                  return ex2x2(ffma2(make_float2(y[i], y[i + 1]), kt2, nLq2));
                else if constexpr (QK == Q_PROBS_T1)
                  return fmul2(make_float2(y[i], y[i + 1]), make_float2(invZq, invZq));
                else
                  return make_float2(q_of<QK>(y[i], kt, invT, negLq, invZq),
                                     q_of<QK>(y[i + 1], kt, invT, negLq, invZq));
              };
              if constexpr (kR) {
  #pragma unroll
                for (int i = 0; i < 8; i += 2) {
                  const float2 p = ex2x2(ffma2(make_float2(x[i], x[i + 1]), kt2, nLp2));
                  const float2 q = q2_of(i);
                  const float2 mn = make_float2(fminf(p.x, q.x), fminf(p.y, q.y));
                  acc_a2 = fadd2(acc_a2, mn);
                  acc_r2 = fadd2(acc_r2, ffma2(mn, make_float2(-1.f, -1.f), p));
                }
              } else if constexpr (QK == Q_LOGITS) {
                // min(p, q) = 2^min(log2 p, log2 q): one exponential
  #pragma unroll
                for (int i = 0; i < 8; i += 2) {
                  const float2 lp = ffma2(make_float2(x[i], x[i + 1]), kt2, nLp2);
                  const float2 lq = ffma2(make_float2(y[i], y[i + 1]), kt2, nLq2);
                  acc_a2 = fadd2(acc_a2, ex2x2(make_float2(fminf(lp.x, lq.x), fminf(lp.y, lq.y))));
                }
              } else {
  #pragma unroll
                for (int i = 0; i < 8; i += 2) {
                  const float2 p = ex2x2(ffma2(make_float2(x[i], x[i + 1]), kt2, nLp2));
                  const float2 q = q2_of(i);
                  acc_a2 = fadd2(acc_a2, make_float2(fminf(p.x, q.x), fminf(p.y, q.y)));
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[stg]);
          if (++stg == NS) {
            stg = 0;
            ++round;
          }
        }
      };
      using Yes = std::true_type;
      using No = std::false_type;
      auto with_b = [&](auto fA, auto fQ) {
        if (qb < 0) chunk_loop(fA, fQ, No{}, No{});
        else if (needR) chunk_loop(fA, fQ, Yes{}, Yes{});
        else chunk_loop(fA, fQ, Yes{}, No{});
      };
      // pass A: the target row unless its normaliser is given, the draft
      // row unless its normaliser is given (or the row has none)
      const bool pA = hA && !plse, pQ = hA && qa >= 0 && !qlse;
      if (pA && pQ) with_b(Yes{}, Yes{});
      else if (pA) with_b(Yes{}, No{});
      else if (pQ) with_b(No{}, Yes{});
      else with_b(No{}, No{});

      // 5. CTA reductions; alpha partial of row j - 1; exchange
      const float acc_a = acc_a2.x + acc_a2.y, acc_r = acc_r2.x + acc_r2.y;
      if constexpr (QK == Q_PROBS_T1) zq += zq2.x + zq2.y;
      {
        const int pb = j & 1;
        const MaxSum A = warp_ms(MaxSum{m, z});
        float w2 = 0.f, w3;
        if (QK == Q_PROBS_T1) {
          w3 = warp_sum(zq);
        } else {
          const MaxSum Bq = warp_ms(MaxSum{mq, zq});
          w2 = Bq.m;
          w3 = Bq.z;
        }
        const float aw = warp_sum(acc_a), rw = warp_sum(acc_r);
        if (lane == 0) {
          sm.wst[pb][warp] = make_float4(A.m, A.z, w2, w3);
          sm.wab[pb][warp] = make_float2(aw, rw);
        }
        named_sync(kBar, kCT);
        if (warp == 0) {
          const float4 v = (lane < kCW) ? sm.wst[pb][lane]
                                        : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
          const float2 ab = (lane < kCW) ? sm.wab[pb][lane] : make_float2(0.f, 0.f);
          MaxSum A2{v.x, v.y}, B2{v.z, v.w};
          float z1 = (lane < kCW) ? v.w : 0.f, aa = ab.x, rr = ab.y;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) {
            A2 = ms_combine(A2, MaxSum{__shfl_xor_sync(0xffffffffu, A2.m, o),
                                       __shfl_xor_sync(0xffffffffu, A2.z, o)});
            if (QK == Q_PROBS_T1) {
              z1 += __shfl_xor_sync(0xffffffffu, z1, o);
            } else {
              B2 = ms_combine(B2, MaxSum{__shfl_xor_sync(0xffffffffu, B2.m, o),
                                         __shfl_xor_sync(0xffffffffu, B2.z, o)});
            }
            aa += __shfl_xor_sync(0xffffffffu, aa, o);
            rr += __shfl_xor_sync(0xffffffffu, rr, o);
          }
          const float4 stats = make_float4(
              __shfl_sync(0xffffffffu, A2.m, 0), __shfl_sync(0xffffffffu, A2.z, 0),
              QK == Q_PROBS_T1 ? 0.f : __shfl_sync(0xffffffffu, B2.m, 0),
              QK == Q_PROBS_T1 ? __shfl_sync(0xffffffffu, z1, 0) : __shfl_sync(0xffffffffu, B2.z, 0));
          const float4 resid = make_float4(__shfl_sync(0xffffffffu, rr, 0), 0.f, 0.f, 0.f);
          if (lane == 0 && qb >= 0) a.alpha_part[ub * kAlphaSlots + rank] = aa;
          const int xs = j & 3;
          if (lane == 0) mbar_expect_tx(&sm.xbar[xs], (uint32_t)C * 32u);
          if (lane < C) {
            const uint32_t bar = mapa(smem_u32(&sm.xbar[xs]), (uint32_t)lane);
            st_async_v4(mapa(smem_u32(&sm.xslot[xs][rank][0]), (uint32_t)lane), stats, bar);
            st_async_v4(mapa(smem_u32(&sm.xslot[xs][rank][1]), (uint32_t)lane), resid, bar);
          }
        }
      }
      q_prev = qa;
      q_cur = q_next;
      u_prev2 = u_prev;
      u_prev = u_cur;
      u_cur = u_next;
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still push to it
}

// The walk: one cluster of C CTAs per sequence (CTA `rank` owns the same
// vocabulary slice as in the streaming kernel).  Acceptance masses (alpha
// partials summed in rank order); then, from the root, follow the accepted
// children.  A row whose recursion is pending gets a pass over its logits
// for each new C (mass of max(0, p - C q), summed over the cluster) until a
// child is accepted or none is left.  The row where the walk stops draws its
// token by inverse CDF in vocabulary order: slice, 4096-logit chunk,
// 256-logit warp segment, lane, element.
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;

constexpr int kMaxW = 8;  // CTAs per sequence in the walk

struct WalkSmem {
  Meta rec;                           // record of the row the walk is at
  int child[SPEC_MAX_TREE_NODES + 1];  // each row's outcome (RowOut::child)
  float wsum[kMaxTiles][kWalkWarps];  // per (chunk, warp) masses of the draw
  float red[kWalkWarps];
  float xs[2][kMaxW];                 // cluster exchange slots (by parity)
  float xm[2][kMaxW];                 //   (maxima of a normaliser exchange)
  RowOut st;                          // walk state (thread 0 writes)
  int act;                            // 0 done, 1 pass, 2 draw
  int rr, len, rsel, tile, wsel;
  int rec_row;                        // row whose record is in `rec` (-1: none)
  float t;
};

template <typename TT, typename TD, int QK>
__global__ void __launch_bounds__(kWalkThreads) stream_walk(StreamParams P) {
  __shared__ WalkSmem ws;
  // a programmatic dependent of unit_stream: nothing read before it is done
  grid_dependency_wait();
  const VerifyShape& s = P.s;
  const VerifyArgs& a = P.a;
  const int C = P.wC;  // the walk's own split of the vocabulary
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = s.n, V = s.V;
  const int64_t u0 = (int64_t)b * (n + 1);
  const float kt = P.kt, invT = P.invT;
  const int r0 = (int)rank * P.wslice;
  const int len = max(0, min(P.wslice, V - r0));
  const int nch = (len + kCH - 1) / kCH;
  for (int r = tid; r <= n; r += kWalkThreads) ws.child[r] = a.rowout[u0 + r].child;
  if (rank == 0) {
    for (int r = tid; r <= n; r += kWalkThreads) {
      const int64_t row = u0 + r;
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
        for (int k = 0; k < P.C; ++k) m += a.alpha_part[row * kAlphaSlots + k];
      }
      if (s.chain) {
        if (r < n) a.mass[(int64_t)b * n + r] = m;
      } else {
        a.mass[row] = m;
      }
    }
  }
  int xe = 0;  // cluster exchanges so far
  // CTA sum of every thread's `v`, exchanged: the cluster total (the same
  // in every CTA; per-rank totals stay in ws.xs).
  auto reduce_exchange = [&](float v) -> float {
    v = warp_sum(v);
    if (lane == 0) ws.red[warp] = v;
    __syncthreads();
    if (warp == 0) {
      float t = (lane < kWalkWarps) ? ws.red[lane] : 0.f;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (lane < C) {  // this CTA's total into every CTA's slot `rank`
        const uint32_t dst = mapa(smem_u32(&ws.xs[xe & 1][rank]), (uint32_t)lane);
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(t) : "memory");
      }
    }
    cluster_sync();
    float tot = 0.f;
    for (int i = 0; i < C; ++i) tot += ws.xs[xe & 1][i];
    ++xe;
    return tot;
  };
  // Sum over this CTA's slice of row u of max(0, p - Cx q) (p when Cx = 0),
  // optionally keeping the per (chunk, warp) masses; the cluster total
  // comes back from exchange number `xe`.
  auto pass = [&](int64_t u, int qr, float Cx, const RowOut& st, bool keep) -> float {
    const TT* tr = reinterpret_cast<const TT*>(a.target) + u * (int64_t)V + r0;
    const TD* dr = (Cx != 0.f && qr >= 0)
                       ? reinterpret_cast<const TD*>(a.draft) + (u0 / (n + 1) * s.R + qr) * V + r0
                       : nullptr;
    const float nLp = -st.Lp, nLq = -st.Lq, iZ = st.invZq;
    float acc = 0.f;
    constexpr int kIn = 2 * inflight<TT, TD>();
    for (int c0 = 0; c0 < nch; c0 += kIn) {
      Raw8<TT> xt[kIn];
      Raw8<TD> xd[kIn];
#pragma unroll
      for (int v = 0; v < kIn; ++v) {
        const int e = (c0 + v) * kCH + tid * kEPT;
        if (c0 + v < nch && e < len) {
          ldg_raw<TT>(tr + e, xt[v]);
          if (dr) ldg_raw<TD>(dr + e, xd[v]);
        }
      }
#pragma unroll
      for (int v = 0; v < kIn; ++v) {
        const int e = (c0 + v) * kCH + tid * kEPT;
        float ls = 0.f;
        if (c0 + v < nch && e < len) {
          float x[8], y[8];
          unpack8(xt[v], x);
          if (dr) unpack8(xd[v], y);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float p = ex2(fmaf(x[i], kt, nLp));
            ls += dr ? resid_w(p, q_of<QK>(y[i], kt, invT, nLq, iZ), Cx) : p;
          }
        }
        acc += ls;
        if (keep && c0 + v < nch) {
          const float wsm = warp_sum(ls);
          if (lane == 0) ws.wsum[c0 + v][warp] = wsm;
        }
      }
    }
    return reduce_exchange(acc);
  };

  // Base-2 log normaliser of target row u (a row the streaming kernel did
  // not process): online sums over the CTA's slice, (max, sum) exchanged.
  auto lse_pass = [&](int64_t u) -> float {
    const TT* tr = reinterpret_cast<const TT*>(a.target) + u * (int64_t)V + r0;
    float m = neg_inf(), z = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int e = c * kCH + tid * kEPT;
      if (e < len) {
        Raw8<TT> xt;
        ldg_raw<TT>(tr + e, xt);
        float x[8];
        unpack8(xt, x);
        lazy_sum(x, kt, m, z);
      }
    }
    MaxSum A = warp_ms(MaxSum{m, z});
    if (lane == 0) {
      ws.red[warp] = A.m;
      ws.wsum[0][warp] = A.z;
    }
    __syncthreads();
    if (warp == 0) {
      MaxSum B{(lane < kWalkWarps) ? ws.red[lane] : neg_inf(),
               (lane < kWalkWarps) ? ws.wsum[0][lane] : 0.f};
#pragma unroll
      for (int o = 8; o > 0; o >>= 1)
        B = ms_combine(B, MaxSum{__shfl_xor_sync(0xffffffffu, B.m, o),
                                 __shfl_xor_sync(0xffffffffu, B.z, o)});
      if (lane < C) {
        const uint32_t dm = mapa(smem_u32(&ws.xm[xe & 1][rank]), (uint32_t)lane);
        const uint32_t dz = mapa(smem_u32(&ws.xs[xe & 1][rank]), (uint32_t)lane);
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dm), "f"(B.m) : "memory");
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dz), "f"(B.z) : "memory");
      }
    }
    cluster_sync();
    MaxSum T{ws.xm[xe & 1][0], ws.xs[xe & 1][0]};
    for (int i = 1; i < C; ++i) T = ms_combine(T, MaxSum{ws.xm[xe & 1][i], ws.xs[xe & 1][i]});
    ++xe;
    return T.m + log2f(T.z);
  };

  // walk (thread 0 of every CTA, identical decisions)
  if (tid == 0) {
    ws.rr = 0;
    ws.len = 0;
    ws.act = 0;
    ws.rec_row = -1;
  }
  __syncthreads();
  for (;;) {
    if (tid == 0) {
      int rr = ws.rr, plen = ws.len;
      RowOut st;
      bool have = ws.act == 1;  // continuing a pending row
      if (have) st = ws.st;
      int act = 0;
      for (;;) {
        const int ch = have ? st.child : ws.child[rr];
        if (ch >= 0 && ch < n && plen < n) {
          if (rank == 0) {
            if (!s.chain) a.path_nodes[(int64_t)b * n + plen] = ch;
            a.out_tokens[u0 + plen] = a.node_tokens[(int64_t)b * n + ch];
          }
          ++plen;
          rr = ch + 1;
          have = false;
          continue;
        }
        if (!have) st = a.rowout[u0 + rr];  // the row where the walk stops or waits
        act = (st.child == -2) ? 1 : 2;
        break;
      }
      ws.rr = rr;
      ws.len = plen;
      ws.st = st;
      ws.act = act;
    }
    __syncthreads();
    const int act = ws.act;
    const int64_t ur = u0 + ws.rr;
    if (ws.rr != ws.rec_row) {  // the row's record into shared memory, once
      const uint4* src = reinterpret_cast<const uint4*>(a.meta + ur * (int64_t)P.rec_bytes);
      uint4* dst = reinterpret_cast<uint4*>(&ws.rec);
      for (int i = tid; i < P.rec_bytes / 16; i += kWalkThreads) dst[i] = src[i];
      __syncthreads();
      if (tid == 0) ws.rec_row = ws.rr;
    }
    const Meta* M = &ws.rec;
    const int qr = M->qr;
    RowOut st = ws.st;
    if (act == 1) {
      const float Wn = pass(ur, qr, st.Cn, st, false);
      if (tid == 0) {
        siblings<QK>(*M, P.kidcap, st, Wn, -1.f, true, kt, invT, V);
        if (rank == 0) flag_status(a.status, st.bits & ~ws.st.bits);
        ws.st = st;
      }
      __syncthreads();
      continue;
    }
    // draw at row ur from max(0, p - Cn q), else from max(0, p - Cc q)
    if (isnan(st.Lp)) st.Lp = lse_pass(ur);  // a row without a draft row
    float Cx = st.Cn;
    float tot = pass(ur, qr, Cx, st, true);
    if (!(tot > 0.f) && Cx != 0.f) {
      if (tid == 0 && rank == 0) flag_status(a.status, SPEC_STATUS_RESIDUAL_ZERO);
      Cx = st.Cc;
      tot = pass(ur, qr, Cx, st, true);
    }
    if (tid == 0) {
      const float u = M->u_draw;
      float t = u * tot, run = 0.f;
      int sel = -1, last = -1;
      for (int k = 0; k < C; ++k) {
        const float w = ws.xs[(xe - 1) & 1][k];
        if (w > 0.f) {
          last = k;
          if (sel < 0 && run + w > t) sel = k;
        }
        if (sel < 0) run += w;
      }
      if (sel < 0) {  // rounding: the last slice with mass, its last token with mass
        sel = last;
        t = 3.0e38f;
        run = 0.f;
      }
      ws.rsel = sel;
      ws.t = t - run;
      if (sel < 0 && rank == 0) flag_status(a.status, SPEC_STATUS_CDF_FALLBACK);
    }
    __syncthreads();
    const int rsel = ws.rsel;
    if (rsel == (int)rank) {
      if (warp == 0) {
        float ct = 0.f;
        if (lane < nch)
          for (int w = 0; w < kWalkWarps; ++w) ct += ws.wsum[lane][w];
        float inc = ct;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        float t = ws.t;
        uint32_t cr = __ballot_sync(0xffffffffu, lane < nch && ct > 0.f && inc > t);
        int tc;
        if (cr) {
          tc = __ffs(cr) - 1;
        } else {
          const uint32_t pos = __ballot_sync(0xffffffffu, lane < nch && ct > 0.f);
          tc = pos ? 31 - __clz(pos) : 0;
          t = 3.0e38f;
        }
        t -= __shfl_sync(0xffffffffu, inc - ct, tc);
        const float wv = (lane < kWalkWarps) ? ws.wsum[tc][lane] : 0.f;
        float winc = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, winc, o);
          if (lane >= o) winc += y;
        }
        uint32_t wc = __ballot_sync(0xffffffffu, lane < kWalkWarps && wv > 0.f && winc > t);
        int tw;
        if (wc) {
          tw = __ffs(wc) - 1;
        } else {
          const uint32_t pos = __ballot_sync(0xffffffffu, lane < kWalkWarps && wv > 0.f);
          tw = pos ? 31 - __clz(pos) : 0;
          t = 3.0e38f;
        }
        t -= __shfl_sync(0xffffffffu, winc - wv, tw);
        if (lane == 0) {
          ws.tile = tc;
          ws.wsel = tw;
          ws.t = t;
        }
      }
      __syncthreads();
      if (warp == ws.wsel) {
        const int base = ws.tile * kCH + ws.wsel * 256 + lane * kEPT;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (base < len) {
          const TT* tr = reinterpret_cast<const TT*>(a.target) + ur * (int64_t)V + r0;
          Raw8<TT> xt;
          ldg_raw<TT>(tr + base, xt);
          float x[8], y[8];
          unpack8(xt, x);
          const bool useq = Cx != 0.f && qr >= 0;
          if (useq) {
            const TD* dr = reinterpret_cast<const TD*>(a.draft) + ((int64_t)b * s.R + qr) * V + r0;
            Raw8<TD> xd;
            ldg_raw<TD>(dr + base, xd);
            unpack8(xd, y);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float p = ex2(fmaf(x[i], kt, -st.Lp));
            v[i] = useq ? resid_w(p, q_of<QK>(y[i], kt, invT, -st.Lq, st.invZq), Cx) : p;
          }
        }
        const float ls = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
        float inc = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        float t = ws.t;
        const uint32_t cr = __ballot_sync(0xffffffffu, ls > 0.f && inc > t);
        int tl;
        if (cr) {
          tl = __ffs(cr) - 1;
        } else {
          const uint32_t pos = __ballot_sync(0xffffffffu, ls > 0.f);
          tl = pos ? 31 - __clz(pos) : 0;
          t = 3.0e38f;
        }
        t -= __shfl_sync(0xffffffffu, inc - ls, tl);
        int pick = -1, lastpos = -1;
        float run = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          run += v[i];
          if (v[i] > 0.f) {
            lastpos = i;
            if (pick < 0 && run > t) pick = i;
          }
        }
        if (pick < 0) pick = lastpos;
        pick = __shfl_sync(0xffffffffu, pick, tl);
        if (lane == 0) {
          const int b0 = ws.tile * kCH + ws.wsel * 256;
          const int tok = r0 + b0 + tl * kEPT + (pick < 0 ? 0 : pick);
          const int plen = ws.len;
          a.out_tokens[u0 + plen] = tok;
          if (pick < 0) flag_status(a.status, SPEC_STATUS_CDF_FALLBACK);
        }
      }
    } else if (rsel < 0 && rank == 0 && tid == 0) {
      a.out_tokens[u0 + ws.len] = 0;
    }
    break;
  }
  if (rank == 0 && tid == 0) {
    const int plen = ws.len;
    for (int k = plen + 1; k <= n; ++k) a.out_tokens[u0 + k] = -1;
    if (!s.chain)
      for (int k = plen; k < n; ++k) a.path_nodes[(int64_t)b * n + k] = -1;
    a.count[b] = plen;
  }
  cluster_sync();  // no CTA leaves while a peer may still write to it
}

// L2 that the pass-B re-reads may count on: a cluster's pass A of row j and
// pass B of row j - 1 are one row-time apart, so every cluster keeps one
// row's pass-A bytes (its slices) in L2 until they are read again.  With
// 152 single-CTA clusters a static-tree row (2 + 4 bytes per logit at V =
// 128256) would keep 117 MB in flight and pass B fell out of L2 (the
// kernel took 0.397 ms against 0.253 ms with clusters of 2); an EAGLE-2
// row whose draft normaliser is given keeps only the target row, 39 MB.
constexpr int64_t kL2Keep = 64LL << 20;

// Geometry for rows of V logits with element sizes tsz (target), dsz (draft):
// the smallest cluster whose slices fit the walk's chunk table, and as many
// ring stages as fit kRing.  One CTA per row (no cluster exchange, twice the
// logits per row-time) when there are at least as many rows as SMs and the
// rows' pass-A bytes (passA per logit) in flight fit kL2Keep; otherwise
// clusters of 2 or more.  False when the streaming kernel does not apply (V
// not a multiple of 8, or rows too long).
inline bool geometry(int V, int tsz, int dsz, int* C, int* slice, int* nch, int* stages,
                     int64_t rows = 0, int sms = 0, int passA = 0) {
  if (V <= 0 || V % 8 != 0) return false;
  const int64_t stage = 2LL * kCH * (tsz + dsz);
  const int ns = (int)(kRing / stage);
  if (ns < 2) return false;
  const bool single = sms > 0 && rows >= sms &&
                      (int64_t)sms * V * passA <= kL2Keep;
  for (int c = single ? 1 : 2; c <= kMaxC; c *= 2) {
    const int sl = ((V + c - 1) / c + 7) / 8 * 8;
    const int nc = (sl + kCH - 1) / kCH;
    if (nc > kMaxTiles) continue;
    *C = c;
    *slice = sl;
    *nch = nc;
    *stages = ns < kMaxNS ? ns : kMaxNS;
    return true;
  }
  return false;
}

template <typename TT, typename TD, int QK>
cudaError_t launch_t(StreamParams P, cudaStream_t st) {
  // the shared-memory barrier arrays hold kMaxNS stages and kMaxC ranks
  if (P.stages < 2 || P.stages > kMaxNS || P.C < 1 || P.C > kMaxC) return cudaErrorInvalidValue;
  auto kern = unit_stream<TT, TD, QK>;
  const size_t dyn = (size_t)P.stages * 2 * kCH * (sizeof(TT) + sizeof(TD));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch on row_meta (set for the launch below)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(P.C);
  int maxc = 0;
  e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (maxc < 1) return cudaErrorInvalidConfiguration;
  const int64_t units = P.s.rows();
  P.nclusters = (int)(units < maxc ? units : maxc);
  row_meta<TT, TD><<<(unsigned)((units + 7) / 8), 256, 0, st>>>(P.s, P.a, P.kidcap, P.rec_bytes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(P.nclusters * P.C));
  cfg.numAttrs = 2;
  prof_begin(SPEC_PROF_VERIFY, st);
  e = cudaLaunchKernelEx(&cfg, kern, P);
  prof_end(SPEC_PROF_VERIFY, st);
  if (e != cudaSuccess) return e;
  // walk: as many CTAs per sequence (1..4) as fit the GPU at two CTAs per SM
  // (more made the cluster barriers cost more than the passes gain), at
  // least enough for the draw's chunk table (up to 8)
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  if (e != cudaSuccess) return e;
  int w = 1;
  while (w < 4 && (int64_t)P.s.B * w * 2 <= 2 * sms) w *= 2;
  for (;;) {
    const int sl = ((P.s.V + w - 1) / w + 7) / 8 * 8;
    if ((sl + kCH - 1) / kCH <= kMaxTiles || w == kMaxW) {
      P.wC = w;
      P.wslice = sl;
      break;
    }
    w *= 2;
  }
  if ((P.wslice + kCH - 1) / kCH > kMaxTiles) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute wattr[2];
  wattr[0].id = cudaLaunchAttributeClusterDimension;
  wattr[0].val.clusterDim.x = P.wC;
  wattr[0].val.clusterDim.y = 1;
  wattr[0].val.clusterDim.z = 1;
  // programmatic dependent launch on unit_stream
  wattr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  wattr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t wc = {};
  wc.blockDim = dim3(kWalkThreads);
  wc.gridDim = dim3((unsigned)(P.s.B * P.wC));
  wc.stream = st;
  wc.attrs = wattr;
  wc.numAttrs = 2;
  return cudaLaunchKernelEx(&wc, stream_walk<TT, TD, QK>, P);
}

template <typename TT, typename TD>
cudaError_t launch_dt(const StreamParams& P, cudaStream_t st) {
  if (P.qk == Q_LOGITS) return launch_t<TT, TD, Q_LOGITS>(P, st);
  if (P.qk == Q_PROBS_T1) return launch_t<TT, TD, Q_PROBS_T1>(P, st);
  return launch_t<TT, TD, Q_PROBS_T>(P, st);
}

}  // namespace
}  // namespace stream
}  // namespace sv
