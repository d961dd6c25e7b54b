// Sampled verification with top-k (and optionally top-p) truncation.
//
// The transform of the Leviathan analysis page ("064 · 投机解码", section 二:
// p and q both go through the same temperature / top-k / nucleus transform)
// leaves each row with at most k tokens of positive probability, so after one
// streaming top-k pass over every target and draft row the whole method runs
// on at most 2k candidates per row:
//   * softmax of z / T over the kept tokens; top-p keeps the shortest prefix
//     (probability descending, index ascending) whose mass reaches top_p,
//     at least one token, then renormalises;
//   * alpha = sum over the common support of min(p, q);
//   * children tried in index order, accept iff u < p'(x) / q'(x); after a
//     rejection the residual max(0, p - C q) (the unrolled norm(max(0, p' -
//     q')) recursion of the full-vocabulary kernels);
//   * no child accepted: inverse-CDF draw from the final weights in
//     vocabulary order (a leaf: the bonus token from p).
// Kernels: topk_rows (one CTA per target row and per draft row, one HBM
// pass; a target row's CTA also builds the row's record -- children and
// uniforms, as for the streaming path) and sparse_warp (one warp per row,
// all math on the candidate lists as warp-wide sums and scans; the warp that
// finishes a sequence's last row walks the sequence).
#include "sample_stream.cuh"
#include "topk.cuh"

namespace sv {
namespace {

constexpr int kK = topk::kMaxK;
// topk_rows' dynamic shared memory: the fallback's buffers, whose space also
// holds the group keys of rows of up to gk_slots_for(kTopkSmem) groups per
// thread
constexpr size_t kTopkSmem = (size_t)topk::kWarps * topk::kBufCap * sizeof(topk::Cand);

struct TopkOut {
  int32_t* idx;   // [2 * rows * kK]: target rows, then draft rows
  float* val;
  int32_t* cnt;   // [2 * rows]
};

// blockIdx.x < rows: target row; else the draft row of tree row
// blockIdx.x - rows (none: count 0).
// Five CTAs per SM (at most 48 registers, four 16-byte loads in flight per
// thread): 760 rows resident at once, so a batch of that many rows streams
// in one wave and the per-row tails (bound, rescan, ranking) overlap.
// The target row's CTA also builds the row's record (its last warp, while
// the others rank the candidates) and, for a sequence's first row, clears
// the sequence's counter of finished rows.
template <typename TT, typename TD, bool kVecT, bool kVecD>
__global__ void __launch_bounds__(topk::kThreads, 5) topk_rows(VerifyShape s, VerifyArgs a, int k,
                                                               TopkOut o, int kidcap,
                                                               int rec_bytes, int32_t* seqcnt) {
  extern __shared__ __align__(16) unsigned char smraw[];
  topk::Cand* smem = reinterpret_cast<topk::Cand*>(smraw);
  // the candidate-list kernel may be scheduled as SMs free up; it waits for
  // this grid to finish before it reads anything
  launch_dependents();
  const int64_t rows = s.rows();
  const int64_t i = blockIdx.x;
  const int n = s.n, V = s.V;
  if (i < rows) {
    if (threadIdx.x == 0 && i % (n + 1) == 0) seqcnt[i / (n + 1)] = 0;
    const TT* rp = reinterpret_cast<const TT*>(a.target) + i * (int64_t)V;
    auto record = [&](int lane) {
      stream::row_meta_warp<TT, TD>(s, a, i, lane, kidcap, rec_bytes);
    };
    topk::row_topk_fast<TT, kVecT, 4>(rp, V, k, 1.f, smem, o.idx + i * kK, o.val + i * kK,
                                      o.cnt + i, nullptr, topk::gk_slots_for(kTopkSmem), record);
    return;
  }
  const int64_t u = i - rows;
  const int b = (int)(u / (n + 1));
  const int r = (int)(u - (int64_t)b * (n + 1));
  int q = -1;
  if (s.chain) q = (r < n) ? r : -1;
  else if (a.q_row) q = a.q_row[u];
  if (q < 0 || q >= s.R) {
    if (threadIdx.x == 0) o.cnt[i] = 0;
    return;
  }
  const TD* rp = reinterpret_cast<const TD*>(a.draft) + ((int64_t)b * s.R + q) * V;
  topk::row_topk_fast<TD, kVecD, 4>(rp, V, k, 1.f, smem, o.idx + i * kK, o.val + i * kK,
                                    o.cnt + i, nullptr, topk::gk_slots_for(kTopkSmem));
}

constexpr int kSW = 4;  // rows (warps) per CTA of sparse_warp
constexpr unsigned kFull = 0xffffffffu;

// Sum over the warp, the same value in every lane (taken from lane 0).
__device__ __forceinline__ float wsum(float v) {
  return __shfl_sync(kFull, warp_sum(v), 0);
}
// Inclusive prefix sum of one value per lane.
__device__ __forceinline__ float wscan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Probabilities of a candidate list (raw values, best first; lane l holds
// positions l + 32 i) after the temperature, softmax and top-p steps, written
// to prob[pos] (0 past the cut).  Returns the kept count.
__device__ int warp_transform(const float (&val)[4], int cnt, bool probs, float kt, float invT,
                              float top_p, float* prob, int lane) {
  if (cnt <= 0) return 0;
  float e[4], loc = 0.f;
  float sv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = lane + 32 * i;
    sv[i] = pos < cnt ? (probs ? __fmul_rn(lg2(val[i]), invT) : __fmul_rn(val[i], kt)) : neg_inf();
  }
  const float s0 = __shfl_sync(kFull, sv[0], 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = lane + 32 * i;
    e[i] = (pos < cnt && s0 != neg_inf()) ? ex2(sv[i] - s0) : 0.f;
    loc += e[i];
  }
  const float Z = wsum(loc);
  if (!(Z > 0.f)) {  // no finite logit among the candidates
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lane + 32 * i < cnt) prob[lane + 32 * i] = 0.f;
    return 0;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) e[i] = e[i] / Z;
  int keep = cnt;
  if (top_p < 1.f) {
    // shortest prefix (list order) whose mass reaches top_p, at least one
    float carry = 0.f;
    bool found = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int pos = lane + 32 * i;
      const float c = carry + wscan(e[i], lane);
      const unsigned hit = __ballot_sync(kFull, pos < cnt && c >= top_p);
      if (!found && hit) {
        keep = 32 * i + __ffs(hit);
        found = true;
      }
      carry = __shfl_sync(kFull, c, 31);
    }
    float z2 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) z2 += (lane + 32 * i < keep) ? e[i] : 0.f;
    z2 = wsum(z2);
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = (lane + 32 * i < keep) ? e[i] / z2 : 0.f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (lane + 32 * i < cnt) prob[lane + 32 * i] = e[i];
  return keep;
}

// One warp per tree row: the transform of both candidate lists, the
// acceptance mass, the children's tests and the draw, all as warp-wide sums
// and scans over the at most kK candidates (no block barrier).
template <typename TT, typename TD>
__global__ void __launch_bounds__(32 * kSW) sparse_warp(VerifyShape s, VerifyArgs a, TopkOut o,
                                                        float kt, float invT, int rec_bytes,
                                                        int kidcap, int32_t* seqcnt) {
  constexpr int kRecMax = (16 + 20 * SPEC_MAX_CHILDREN + 15) / 16;  // 16-byte words
  struct WarpMem {
    uint4 rec[kRecMax];          // the row's record
    float pk[kK], qk[kK];        // probabilities, list order
    int32_t tis[kK], dis[kK];    // candidate tokens, list order
    int32_t ptok_v[kK];          // support of p in vocabulary order
    float pv_v[kK], qv_v[kK];    // p and q at those tokens
  };
  __shared__ WarpMem wmem[kSW];
  // launched as a programmatic dependent of topk_rows: nothing it wrote is
  // read before that grid has completed
  grid_dependency_wait();
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int64_t rows = s.rows();
  const int64_t u = (int64_t)blockIdx.x * kSW + wi;
  if (u >= rows) return;  // the whole warp
  WarpMem& m = wmem[wi];
  const int V = s.V;
  {  // the record into shared memory, its loads beside the lists' below
    const uint4* src = reinterpret_cast<const uint4*>(a.meta + u * (int64_t)rec_bytes);
    for (int i = lane; i < rec_bytes / 16; i += 32) m.rec[i] = src[i];
  }
  const stream::Meta* M = reinterpret_cast<const stream::Meta*>(m.rec);
  const float* ukid = reinterpret_cast<const float*>(
      reinterpret_cast<const unsigned char*>(m.rec) + 16 + 16 * kidcap);
  const bool probs = a.prm.draft_kind == SPEC_DRAFT_PROBS;
  const int ct = o.cnt[u], cq = o.cnt[rows + u];
  float tval[4], dval[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = lane + 32 * i;
    tval[i] = pos < ct ? o.val[u * kK + pos] : neg_inf();
    m.tis[pos] = pos < ct ? o.idx[u * kK + pos] : INT_MAX;
    dval[i] = pos < cq ? o.val[(rows + u) * kK + pos] : neg_inf();
    m.dis[pos] = pos < cq ? o.idx[(rows + u) * kK + pos] : -1;
  }
  __syncwarp();
  const bool has_q = M->qr >= 0 && cq > 0;
  const int np = warp_transform(tval, ct, false, kt, invT, a.prm.top_p, m.pk, lane);
  const int nq = has_q ? warp_transform(dval, cq, probs, kt, invT, a.prm.top_p, m.qk, lane) : 0;
  if (lane == 0) {
    uint32_t bad = M->bad;
    if (ct <= 0) bad |= SPEC_STATUS_NAN;
    if (bad) flag_status(a.status, bad);
  }
  __syncwarp();
  // support of p in vocabulary order (tokens are distinct: rank by counting)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = lane + 32 * i;
    if (pos < np) {
      const int t = m.tis[pos];
      int rk = 0;
#pragma unroll 8
      for (int j = 0; j < np; ++j) rk += (m.tis[j] < t) ? 1 : 0;
      float qa = 0.f;
#pragma unroll 8
      for (int j = 0; j < nq; ++j)
        if (m.dis[j] == t) qa = m.qk[j];
      m.ptok_v[rk] = t;
      m.pv_v[rk] = m.pk[pos];
      m.qv_v[rk] = qa;
    }
  }
  __syncwarp();
  auto p_at = [&](int x) -> float {  // at most one match: the sum is exact
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int pos = lane + 32 * i;
      if (pos < np && m.ptok_v[pos] == x) r = m.pv_v[pos];
    }
    return wsum(r);
  };
  auto q_at = [&](int x) -> float {
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int pos = lane + 32 * i;
      if (pos < nq && m.dis[pos] == x) r = m.qk[pos];
    }
    return wsum(r);
  };
  // acceptance mass over the common support
  float al = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = lane + 32 * i;
    if (pos < np) al += fminf(m.pv_v[pos], m.qv_v[pos]);
  }
  const float alpha = wsum(al);

  uint32_t st_bits = 0;
  float Cc = 0.f, W = 1.f, D = 1.f;
  int accepted = -1;
  const int nk = has_q ? M->nk : 0;
  if (M->nk > 0 && !has_q) st_bits |= SPEC_STATUS_BAD_TREE;
  for (int k = 0; k < nk; ++k) {  // every lane takes the same branches
    const int x = M->kid[k].tok;
    bool removed = false;
    for (int i = 0; i < k; ++i) removed |= (M->kid[i].tok == x);
    const bool valid = x >= 0 && x < V;
    float qx = 0.f;
    if (!valid) {
      st_bits |= SPEC_STATUS_TOKEN_RANGE;
    } else {
      const float px = p_at(x);
      qx = q_at(x);
      const float ax = Cc == 0.f ? px : fmaxf(0.f, fmaf(-Cc, qx, px));
      const float qj = removed ? 0.f : qx / D;
      if (qj == 0.f) {
        st_bits |= SPEC_STATUS_QZERO_ACCEPT;
        accepted = M->kid[k].node;
        break;
      }
      if (ukid[k] < (ax / W) / qj) {
        accepted = M->kid[k].node;
        break;
      }
    }
    // rejected: residual max(0, p - Cn q) over the support of p
    const float Cn = Cc + W / D;
    float wl = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int pos = lane + 32 * i;
      if (pos < np) wl += fmaxf(0.f, fmaf(-Cn, m.qv_v[pos], m.pv_v[pos]));
    }
    const float Wn = wsum(wl);
    if (Wn > 0.f) {
      Cc = Cn;
      W = Wn;
    } else {
      st_bits |= SPEC_STATUS_RESIDUAL_ZERO;
    }
    if (valid && !removed) D -= qx;
    if (D <= 0.f) {
      st_bits |= SPEC_STATUS_DRAFT_EXHAUSTED;
      break;
    }
  }
  if (accepted < 0) {
    // inverse CDF of the final weights in vocabulary order
    float w[4], tl = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int pos = lane + 32 * i;
      w[i] = pos < np ? ((Cc == 0.f) ? m.pv_v[pos]
                                     : fmaxf(0.f, fmaf(-Cc, m.qv_v[pos], m.pv_v[pos])))
                      : 0.f;
      tl += w[i];
    }
    const float t = M->u_draw * wsum(tl);
    float carry = 0.f;
    int tok = -1, lastpos = -1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float c = carry + wscan(w[i], lane);
      const unsigned pos_mask = __ballot_sync(kFull, w[i] > 0.f);
      if (pos_mask) lastpos = 32 * i + 31 - __clz(pos_mask);
      const unsigned hit = __ballot_sync(kFull, w[i] > 0.f && c > t);
      if (tok < 0 && hit) tok = m.ptok_v[32 * i + __ffs(hit) - 1];
      carry = __shfl_sync(kFull, c, 31);
    }
    if (tok < 0) {
      tok = lastpos < 0 ? 0 : m.ptok_v[lastpos];
      st_bits |= SPEC_STATUS_CDF_FALLBACK;
    }
    if (lane == 0) a.row_token[u] = tok;
  }
  const int n = s.n;
  const int64_t bq = u / (n + 1);
  if (lane == 0) {
    a.row_child[u] = accepted;
    if (st_bits) flag_status(a.status, st_bits);
    // the row's acceptance mass (NaN for a row without a draft row)
    const int r = (int)(u - bq * (n + 1));
    const float mm = M->qr >= 0 ? alpha : __int_as_float(0x7fc00000);
    if (s.chain) {
      if (r < n) a.mass[bq * n + r] = mm;
    } else {
      a.mass[u] = mm;
    }
  }
  // the warp that finishes a sequence's last row walks the sequence: along
  // the accepted children, then the token drawn where the walk stops
  __threadfence();
  int last = 0;
  if (lane == 0) last = atomicAdd(&seqcnt[bq], 1) == n ? 1 : 0;
  if (!__shfl_sync(kFull, last, 0)) return;
  __threadfence();
  const int64_t row0 = bq * (n + 1);
  int32_t* out = a.out_tokens + row0;
  int rr = 0, len = 0;
  if (n < kK) {
    // every row's outcome and every node's token in one round of loads (the
    // lanes in parallel), then the walk from shared memory
    int32_t* rc = m.ptok_v;  // [n + 1] accepted child per row (free by now)
    int32_t* rt = m.tis;     // [n + 1] token drawn per row
    int32_t* nt = m.dis;     // [n] drafted token per node
    __syncwarp();
    for (int r = lane; r <= n; r += 32) {
      rc[r] = __ldcg(a.row_child + row0 + r);
      rt[r] = __ldcg(a.row_token + row0 + r);
      if (r < n) nt[r] = a.node_tokens[bq * n + r];
    }
    __syncwarp();
    if (lane != 0) return;
    while (true) {
      const int j = rc[rr];
      if (j < 0 || j >= n || len >= n) break;
      if (!s.chain) a.path_nodes[bq * n + len] = j;
      out[len] = nt[j];
      ++len;
      rr = j + 1;
    }
    out[len] = rt[rr];
  } else {  // long sequences: the walk's loads one after another
    if (lane != 0) return;
    while (true) {
      const int j = __ldcg(a.row_child + row0 + rr);
      if (j < 0 || j >= n || len >= n) break;
      if (!s.chain) a.path_nodes[bq * n + len] = j;
      out[len] = a.node_tokens[bq * n + j];
      ++len;
      rr = j + 1;
    }
    out[len] = __ldcg(a.row_token + row0 + rr);
  }
  for (int k = len + 1; k <= n; ++k) out[k] = -1;
  if (!s.chain)
    for (int k = len; k < n; ++k) a.path_nodes[bq * n + k] = -1;
  a.count[bq] = len;
}

template <typename TT, typename TD>
cudaError_t launch_sparse_t(const VerifyShape& s, const VerifyArgs& a, int k, cudaStream_t st) {
  const int64_t rows = s.rows();
  TopkOut o{a.topk_idx, a.topk_val, a.topk_cnt};
  // per-sequence counters of finished rows live in the streaming path's work
  // list (unused here); the row records skip that list
  int32_t* seqcnt = a.qlist;
  if (!seqcnt) return cudaErrorInvalidValue;
  VerifyArgs am = a;
  am.qlist = nullptr;
  const int kidcap = meta_kidcap(s.chain), rec = meta_rec_bytes(s.chain);
  const bool vt = ((uintptr_t)a.target % 16 == 0) && ((int64_t)s.V * sizeof(TT) % 16 == 0) &&
                  (s.V % 8 == 0);
  const bool vd = a.draft && ((uintptr_t)a.draft % 16 == 0) &&
                  ((int64_t)s.V * sizeof(TD) % 16 == 0) && (s.V % 8 == 0);
  const size_t smem = kTopkSmem;
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the largest shared-memory carveout, so that five CTAs fit on an SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(2 * rows), topk::kThreads, smem, st>>>(s, am, k, o, kidcap, rec, seqcnt);
    return cudaGetLastError();
  };
  cudaError_t e;
  prof_begin(SPEC_PROF_VERIFY, st);
  if (vt && vd) e = launch(topk_rows<TT, TD, true, true>);
  else if (vt) e = launch(topk_rows<TT, TD, true, false>);
  else if (vd) e = launch(topk_rows<TT, TD, false, true>);
  else e = launch(topk_rows<TT, TD, false, false>);
  prof_end(SPEC_PROF_VERIFY, st);
  if (e != cudaSuccess) return e;
  const float T = a.prm.temperature;
  // a programmatic dependent launch: its CTAs take the SMs topk_rows leaves
  // and start the moment that grid completes, instead of after a launch
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kSW - 1) / kSW));
  cfg.blockDim = dim3(32 * kSW);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_warp<TT, TD>, s, a, o, kLog2e / T, 1.f / T, rec, kidcap,
                            seqcnt);
}

}  // namespace

cudaError_t launch_sparse(const VerifyShape& s, const VerifyArgs& a, int k, cudaStream_t st) {
  if (s.B == 0) return cudaSuccess;
  if (a.dt_target == SPEC_BF16) {
    if (a.dt_draft == SPEC_BF16) return launch_sparse_t<uint16_t, uint16_t>(s, a, k, st);
    return launch_sparse_t<uint16_t, float>(s, a, k, st);
  }
  if (a.dt_draft == SPEC_BF16) return launch_sparse_t<float, uint16_t>(s, a, k, st);
  return launch_sparse_t<float, float>(s, a, k, st);
}

}  // namespace sv
