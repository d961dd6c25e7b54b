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
// pass), row_meta (children and uniforms, shared with the streaming path),
// sparse_units (one CTA per row, all math on the candidate lists),
// sparse_walk.
#include "sample_stream.cuh"
#include "topk.cuh"

namespace sv {
namespace {

constexpr int kK = topk::kMaxK;

struct TopkOut {
  int32_t* idx;   // [2 * rows * kK]: target rows, then draft rows
  float* val;
  int32_t* cnt;   // [2 * rows]
};

// blockIdx.x < rows: target row; else the draft row of tree row
// blockIdx.x - rows (none: count 0).
template <typename TT, typename TD, bool kVecT, bool kVecD>
__global__ void __launch_bounds__(topk::kThreads) topk_rows(VerifyShape s, VerifyArgs a, int k,
                                                            TopkOut o) {
  extern __shared__ __align__(16) unsigned char smraw[];
  topk::Cand* smem = reinterpret_cast<topk::Cand*>(smraw);
  const int64_t rows = s.rows();
  const int64_t i = blockIdx.x;
  const int n = s.n, V = s.V;
  if (i < rows) {
    const TT* rp = reinterpret_cast<const TT*>(a.target) + i * (int64_t)V;
    topk::row_topk_fast<TT, kVecT>(rp, V, k, 1.f, smem, o.idx + i * kK, o.val + i * kK, o.cnt + i,
                              nullptr);
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
  topk::row_topk_fast<TD, kVecD>(rp, V, k, 1.f, smem, o.idx + i * kK, o.val + i * kK, o.cnt + i,
                            nullptr);
}

// Probabilities of a candidate list (raw values, best first) after the
// temperature, softmax and top-p steps; entries past the cut get 0.
// Thread 0 only; deterministic order.
__device__ int transform_list(const float* val, int cnt, bool probs, float kt, float invT,
                              float top_p, float* prob) {
  if (cnt <= 0) return 0;
  float s0;
  for (int i = 0; i < cnt; ++i) {
    const float sv = probs ? __fmul_rn(lg2(val[i]), invT) : __fmul_rn(val[i], kt);
    if (i == 0) s0 = sv;
    prob[i] = (s0 == neg_inf()) ? 0.f : ex2(sv - s0);
  }
  float Z = 0.f;
  for (int i = 0; i < cnt; ++i) Z += prob[i];
  if (!(Z > 0.f)) {  // no finite logit among the candidates
    for (int i = 0; i < cnt; ++i) prob[i] = 0.f;
    return 0;
  }
  for (int i = 0; i < cnt; ++i) prob[i] = prob[i] / Z;
  int keep = cnt;
  if (top_p < 1.f) {
    float c = 0.f;
    keep = cnt;
    for (int i = 0; i < cnt; ++i) {
      c += prob[i];
      if (c >= top_p) {
        keep = i + 1;
        break;
      }
    }
    float z2 = 0.f;
    for (int i = 0; i < keep; ++i) z2 += prob[i];
    for (int i = 0; i < cnt; ++i) prob[i] = (i < keep) ? prob[i] / z2 : 0.f;
  }
  return keep;
}

template <typename TT, typename TD>
__global__ void __launch_bounds__(kK) sparse_units(VerifyShape s, VerifyArgs a, TopkOut o,
                                                   float kt, float invT, int rec_bytes,
                                                   int kidcap) {
  __shared__ float pk[kK], qk[kK];          // probabilities, list order
  __shared__ int ptok_v[kK];                // support of p in vocabulary order
  __shared__ float pv_v[kK], qv_v[kK];      // p and q at those tokens
  __shared__ float tvs[kK], dvs[kK];        // candidate values (target, draft)
  __shared__ int32_t tis[kK], dis[kK];      // candidate tokens
  __shared__ int s_np, s_nq;
  const int64_t u = blockIdx.x;
  const int64_t rows = s.rows();
  const int tid = threadIdx.x;
  const int V = s.V;
  const stream::Meta* M = reinterpret_cast<const stream::Meta*>(a.meta + u * (int64_t)rec_bytes);
  const float* ukid = reinterpret_cast<const float*>(a.meta + u * (int64_t)rec_bytes + 16 +
                                                     16 * kidcap);
  const bool probs = a.prm.draft_kind == SPEC_DRAFT_PROBS;
  const int ct = o.cnt[u], cq = o.cnt[rows + u];
  const float* tv = o.val + u * kK;
  const int32_t* ti = o.idx + u * kK;
  const float* dv = o.val + (rows + u) * kK;
  const int32_t* di = o.idx + (rows + u) * kK;
  const bool has_q = M->qr >= 0 && cq > 0;
  // the candidate lists into shared memory (one element per thread: at most
  // kK each), so that the serial steps below read no global memory
  if (tid < ct) {
    tvs[tid] = tv[tid];
    tis[tid] = ti[tid];
  }
  if (tid < cq) {
    dvs[tid] = dv[tid];
    dis[tid] = di[tid];
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t bad = M->bad;
    if (ct <= 0) bad |= SPEC_STATUS_NAN;
    s_np = transform_list(tvs, ct, false, kt, invT, a.prm.top_p, pk);
    s_nq = has_q ? transform_list(dvs, cq, probs, kt, invT, a.prm.top_p, qk) : 0;
    if (bad) flag_status(a.status, bad);
  }
  __syncthreads();
  const int np = s_np, nq = s_nq;
  // support of p in vocabulary order (tokens are distinct: rank by counting)
  if (tid < np) {
    const int t = tis[tid];
    int rk = 0;
    for (int j = 0; j < np; ++j) rk += (tis[j] < t) ? 1 : 0;
    float qa = 0.f;
    for (int j = 0; j < nq; ++j)
      if (dis[j] == t) qa = qk[j];
    ptok_v[rk] = t;
    pv_v[rk] = pk[tid];
    qv_v[rk] = qa;
  }
  __syncthreads();
  if (tid != 0) return;

  auto p_at = [&](int x) -> float {
    int lo = 0, hi = np - 1;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (ptok_v[mid] == x) return pv_v[mid];
      if (ptok_v[mid] < x) lo = mid + 1;
      else hi = mid - 1;
    }
    return 0.f;
  };
  auto q_at = [&](int x) -> float {
    for (int j = 0; j < nq; ++j)
      if (dis[j] == x) return qk[j];
    return 0.f;
  };
  // acceptance mass over the common support
  float alpha = 0.f;
  for (int i = 0; i < np; ++i) alpha += fminf(pv_v[i], qv_v[i]);
  if (M->qr >= 0) a.alpha_part[u * kAlphaSlots] = alpha;

  uint32_t st_bits = 0;
  float Cc = 0.f, W = 1.f, D = 1.f;
  int accepted = -1;
  const int nk = has_q ? M->nk : 0;
  if (M->nk > 0 && !has_q) st_bits |= SPEC_STATUS_BAD_TREE;
  for (int k = 0; k < nk; ++k) {
    const int x = M->kid[k].tok;
    bool removed = false;
    for (int i = 0; i < k; ++i) removed |= (M->kid[i].tok == x);
    if (x < 0 || x >= V) {
      st_bits |= SPEC_STATUS_TOKEN_RANGE;
    } else {
      const float px = p_at(x), qx = q_at(x);
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
    float Wn = 0.f;
    for (int i = 0; i < np; ++i) Wn += fmaxf(0.f, fmaf(-Cn, qv_v[i], pv_v[i]));
    if (Wn > 0.f) {
      Cc = Cn;
      W = Wn;
    } else {
      st_bits |= SPEC_STATUS_RESIDUAL_ZERO;
    }
    if (x >= 0 && x < V && !removed) D -= q_at(x);
    if (D <= 0.f) {
      st_bits |= SPEC_STATUS_DRAFT_EXHAUSTED;
      break;
    }
  }
  if (accepted < 0) {
    float tot = 0.f;
    for (int i = 0; i < np; ++i) tot += (Cc == 0.f) ? pv_v[i] : fmaxf(0.f, fmaf(-Cc, qv_v[i], pv_v[i]));
    const float t = M->u_draw * tot;
    float c = 0.f;
    int tok = -1, last = -1;
    for (int i = 0; i < np; ++i) {
      const float w = (Cc == 0.f) ? pv_v[i] : fmaxf(0.f, fmaf(-Cc, qv_v[i], pv_v[i]));
      if (w > 0.f) last = ptok_v[i];
      c += w;
      if (w > 0.f && c > t) {
        tok = ptok_v[i];
        break;
      }
    }
    if (tok < 0) {
      tok = last < 0 ? 0 : last;
      st_bits |= SPEC_STATUS_CDF_FALLBACK;
    }
    a.row_token[u] = tok;
  }
  a.row_child[u] = accepted;
  if (st_bits) flag_status(a.status, st_bits);
}

// Per row: acceptance mass; per sequence (row 0's thread): the walk along
// accepted children and the token drawn at the row where it stops.
__global__ void sparse_walk(VerifyShape s, VerifyArgs a) {
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
  const float m = has_q ? a.alpha_part[row * kAlphaSlots] : __int_as_float(0x7fc00000);
  if (s.chain) {
    if (r < n) a.mass[(int64_t)b * n + r] = m;
  } else {
    a.mass[row] = m;
  }
  if (r != 0) return;
  int32_t* out = a.out_tokens + row;
  int rr = 0, len = 0;
  while (true) {
    const int j = a.row_child[row + rr];
    if (j < 0 || j >= n || len >= n) break;
    if (!s.chain) a.path_nodes[(int64_t)b * n + len] = j;
    out[len] = a.node_tokens[(int64_t)b * n + j];
    ++len;
    rr = j + 1;
  }
  out[len] = a.row_token[row + rr];
  for (int k = len + 1; k <= n; ++k) out[k] = -1;
  if (!s.chain)
    for (int k = len; k < n; ++k) a.path_nodes[(int64_t)b * n + k] = -1;
  a.count[b] = len;
}

template <typename TT, typename TD>
cudaError_t launch_sparse_t(const VerifyShape& s, const VerifyArgs& a, int k, cudaStream_t st) {
  const int64_t rows = s.rows();
  TopkOut o{a.topk_idx, a.topk_val, a.topk_cnt};
  const bool vt = ((uintptr_t)a.target % 16 == 0) && ((int64_t)s.V * sizeof(TT) % 16 == 0) &&
                  (s.V % 8 == 0);
  const bool vd = a.draft && ((uintptr_t)a.draft % 16 == 0) &&
                  ((int64_t)s.V * sizeof(TD) % 16 == 0) && (s.V % 8 == 0);
  const size_t smem = (size_t)topk::kWarps * topk::kBufCap * sizeof(topk::Cand);
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(2 * rows), topk::kThreads, smem, st>>>(s, a, k, o);
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
  const int kidcap = meta_kidcap(s.chain), rec = meta_rec_bytes(s.chain);
  stream::row_meta<TT, TD><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(s, a, kidcap, rec);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float T = a.prm.temperature;
  sparse_units<TT, TD><<<(unsigned)rows, kK, 0, st>>>(s, a, o, kLog2e / T, 1.f / T, rec, kidcap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sparse_walk<<<(unsigned)((rows + 127) / 128), 128, 0, st>>>(s, a);
  return cudaGetLastError();
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
