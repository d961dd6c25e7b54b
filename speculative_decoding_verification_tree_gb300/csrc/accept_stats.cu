// spec_accept_stats: acceptance records over verification outcomes.
//
// Three records the pages ask a deployment to keep: the distribution of the
// accepted length per round ("064 · 投机解码", section 五), the acceptance
// rate of drafted tokens by tree position and depth (EAGLE-2 notes §3.1,
// Fig. 5) and by interval of the draft model's confidence (§3.2, Fig. 6).
// A drafted token is tested iff its parent is the root or on the accepted
// path and no sibling with a lower index was accepted (the tree rule tries
// siblings in node order, EAGLE-2 notes §2.2); it is accepted iff it is on
// the path.  A chain is the tree whose node k has parent k - 1.
//
// A tested node's parent is the root or the path node at some position i,
// and a path node at position i has depth i + 1, so a tested node's depth is
// 1 (child of the root) or i + 2: no walk up the tree is needed.
//
// Layout of the work.  Up to 64 drafted tokens per round (static and EAGLE-2
// trees, chains), one warp takes a round: each lane owns nodes lane and
// lane + 32, issues all of the round's loads (count, parents, path, and
// confidences) at once, checks the path with shuffles and records path
// positions in a per-warp shared-memory table, so the rounds of a batch run
// in parallel with no block barrier.  Larger trees take a whole CTA per
// round with the same steps in shared memory.  Either way a round's
// counts go into per-CTA shared-memory counters, and those reach the
// caller's int64 / double records with one global atomic per nonzero entry
// when the CTA ends.  The records accumulate across calls.
#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kWarpNodes = 64;      // rounds of up to this many nodes: one warp
constexpr int kStatsWarps = 8;      // warps per CTA in the warp-per-round kernel
constexpr unsigned kFull = 0xffffffffu;

// Shared-memory plan of one CTA (32-bit words, then the 8-byte sums).
struct StatsSmem {
  int n, nbins;
  bool calib;
  // per-round tables: CTA mode par/pos/acc, warp mode pos/acc per warp
  int o_par, o_pos, o_acc;
  // counters (contiguous from o_len to o_inv)
  int o_len, o_nt, o_na, o_dt, o_da, o_ct, o_ca, o_inv;
  int words;
  size_t bytes() const {
    size_t b = ((size_t)words * 4 + 7) & ~(size_t)7;
    return b + (calib ? (size_t)nbins * 8 : 0);
  }
};

inline StatsSmem plan(int n, int nbins, bool tree, bool calib, bool warp) {
  StatsSmem s{};
  s.n = n;
  s.nbins = nbins;
  s.calib = calib;
  int w = 0;
  auto take = [&](int k) {
    const int o = w;
    w += k;
    return o;
  };
  if (tree && warp) {
    s.o_pos = take(kStatsWarps * kWarpNodes);
    s.o_acc = take(kStatsWarps * (kWarpNodes + 2));  // [0] root, [j + 1] node j
  } else if (tree) {
    s.o_par = take(n);
    s.o_pos = take(n);
    s.o_acc = take(n + 1);
  }
  s.o_len = take(n + 1);
  s.o_nt = take(n);
  s.o_na = take(n);
  s.o_dt = take(n);
  s.o_da = take(n);
  s.o_ct = calib ? take(nbins) : 0;
  s.o_ca = calib ? take(nbins) : 0;
  s.o_inv = take(1);
  s.words = w;
  return s;
}

// Per-CTA counters in shared memory.
struct Counters {
  uint32_t *len, *nt, *na, *dt, *da, *ct, *ca, *inv;
  double* cs;
  int nbins;
  bool calib;

  __device__ Counters(uint32_t* smem, const StatsSmem& L, bool has_conf) {
    len = smem + L.o_len;
    nt = smem + L.o_nt;
    na = smem + L.o_na;
    dt = smem + L.o_dt;
    da = smem + L.o_da;
    ct = smem + L.o_ct;
    ca = smem + L.o_ca;
    inv = smem + L.o_inv;
    cs = reinterpret_cast<double*>(smem + ((L.words + 1) & ~1));
    nbins = L.nbins;
    calib = L.calib && has_conf;
    for (int i = threadIdx.x; i <= L.o_inv - L.o_len; i += blockDim.x) len[i] = 0;
    if (calib)
      for (int i = threadIdx.x; i < nbins; i += blockDim.x) cs[i] = 0.0;
  }

  // one tested token: node j at depth dep, confidence c (used only if calib)
  __device__ __forceinline__ void add(int j, int dep, bool acc, float c) {
    atomicAdd(&nt[j], 1u);
    atomicAdd(&dt[dep - 1], 1u);
    if (acc) {
      atomicAdd(&na[j], 1u);
      atomicAdd(&da[dep - 1], 1u);
    }
    if (!calib) return;
    float v = c;
    if (v != v) return;  // NaN: not binned
    v = fminf(fmaxf(v, 0.f), 1.f);
    const int k = min((int)floorf(__fmul_rn(v, (float)nbins)), nbins - 1);
    atomicAdd(&ct[k], 1u);
    if (acc) atomicAdd(&ca[k], 1u);
    atomicAdd(&cs[k], (double)v);
  }

  // after a final __syncthreads: nonzero entries to the caller's records
  __device__ void flush(const spec_accept_stats_t& out, int n) const {
    flush1(out.len_hist, len, n + 1);
    flush1(out.node_tested, nt, n);
    flush1(out.node_accepted, na, n);
    flush1(out.depth_tested, dt, n);
    flush1(out.depth_accepted, da, n);
    if (calib) {
      flush1(out.calib_tested, ct, nbins);
      flush1(out.calib_accepted, ca, nbins);
      if (out.calib_conf_sum)
        for (int i = threadIdx.x; i < nbins; i += blockDim.x)
          if (ct[i]) atomicAdd(out.calib_conf_sum + i, cs[i]);
    }
    flush1(out.invalid, inv, 1);
  }

  __device__ static void flush1(int64_t* dst, const uint32_t* src, int k) {
    if (!dst) return;
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      if (src[i])
        atomicAdd(reinterpret_cast<unsigned long long*>(dst + i), (unsigned long long)src[i]);
  }
};

// One warp per round, n <= 64.
template <bool kTree>
__global__ void __launch_bounds__(kStatsWarps * 32)
    accept_stats_warp(const int32_t* __restrict__ count, const int32_t* __restrict__ parent,
                      const int32_t* __restrict__ path, const float* __restrict__ conf, int B,
                      StatsSmem L, spec_accept_stats_t out) {
  extern __shared__ __align__(16) uint32_t smem[];
  Counters C(smem, L, conf != nullptr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* s_pos = reinterpret_cast<int32_t*>(smem + L.o_pos) + warp * kWarpNodes;
  int32_t* s_acc = reinterpret_cast<int32_t*>(smem + L.o_acc) + warp * (kWarpNodes + 2);
  const int n = L.n;
  const int j0 = lane, j1 = lane + 32;
  __syncthreads();

  for (int b = blockIdx.x * kStatsWarps + warp; b < B; b += gridDim.x * kStatsWarps) {
    const int64_t row = (int64_t)b * n;
    // every load of the round at once (the rows are [B, n], fully allocated)
    const int len = count[b];
    int p0 = j0 - 1, p1 = j1 - 1;  // parents (chain: the previous token)
    int v0 = j0, v1 = j1;          // path positions j0, j1 (chain: 0, 1, ...)
    if (kTree) {
      p0 = j0 < n ? parent[row + j0] : -1;
      p1 = j1 < n ? parent[row + j1] : -1;
      v0 = j0 < n ? path[row + j0] : -1;
      v1 = j1 < n ? path[row + j1] : -1;
    }
    const bool calib = C.calib;
    const float c0 = calib && j0 < n ? conf[row + j0] : 0.f;
    const float c1 = calib && j1 < n ? conf[row + j1] : 0.f;

    bool bad = len < 0 || len > n;
    if (kTree) {
      const bool pb = (j0 < n && (p0 < -1 || p0 >= j0)) || (j1 < n && (p1 < -1 || p1 >= j1));
      bad = __any_sync(kFull, bad || pb);
      if (!bad) {
        s_pos[j0] = -1;
        s_pos[j1] = -1;
        s_acc[j0] = n;  // no accepted child
        s_acc[j1] = n;
        if (lane < 2) s_acc[kWarpNodes + lane] = n;
        __syncwarp();
        // path position i = lane + 32 h holds node v; its parent must be the
        // previous path node (the root for i = 0)
        const int up0 = __shfl_up_sync(kFull, v0, 1), last0 = __shfl_sync(kFull, v0, 31);
        const int up1 = __shfl_up_sync(kFull, v1, 1);
        bool pbad = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = lane + 32 * h;
          const int v = h ? v1 : v0;
          const int prev = lane ? (h ? up1 : up0) : (h ? last0 : -1);
          // parent of v, from the lane that owns node v
          const int s = (v >= 0 && v < n) ? v : 0;
          const int a = __shfl_sync(kFull, p0, s & 31), c = __shfl_sync(kFull, p1, s & 31);
          const int pv = s < 32 ? a : c;
          if (i < len) {
            if (v < 0 || v >= n || prev < -1 || prev >= n || pv != prev) {
              pbad = true;
            } else {
              s_pos[v] = i;
              s_acc[prev + 1] = v;
            }
          }
        }
        bad = __any_sync(kFull, pbad);
        __syncwarp();
      }
    }
    if (!bad) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        if (j >= n) continue;
        const int pj = h ? p1 : p0;
        bool tested, acc;
        int dep;
        if (kTree) {
          const int ppos = pj < 0 ? -1 : s_pos[pj];
          tested = (pj < 0 || ppos >= 0) && j <= s_acc[pj + 1];
          acc = s_pos[j] >= 0;
          dep = ppos + 2;  // root child: 1; child of path position i: i + 2
        } else {
          tested = j <= len;
          acc = j < len;
          dep = j + 1;
        }
        if (tested) C.add(j, dep, acc, h ? c1 : c0);
      }
    }
    if (lane == 0) atomicAdd(bad ? C.inv : &C.len[len], 1u);
    __syncwarp();
  }
  __syncthreads();
  C.flush(out, n);
}

// One CTA per round, any n <= SPEC_MAX_TREE_NODES (rounds above 64 nodes).
// A chain (parent == path == NULL) is read as the tree whose node k has
// parent k - 1 and whose path is 0 .. count - 1.
__global__ void __launch_bounds__(256)
    accept_stats_cta(const int32_t* __restrict__ count, const int32_t* __restrict__ parent,
                     const int32_t* __restrict__ path, const float* __restrict__ conf, int B,
                     StatsSmem L, spec_accept_stats_t out) {
  extern __shared__ __align__(16) uint32_t smem[];
  Counters C(smem, L, conf != nullptr);
  int32_t* s_par = reinterpret_cast<int32_t*>(smem + L.o_par);
  int32_t* s_pos = reinterpret_cast<int32_t*>(smem + L.o_pos);
  int32_t* s_acc = reinterpret_cast<int32_t*>(smem + L.o_acc);
  const int n = L.n, tid = threadIdx.x, nt = blockDim.x;
  __syncthreads();

  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int len = count[b];
    const int64_t row = (int64_t)b * n;
    int local_bad = len < 0 || len > n;
    for (int j = tid; j < n; j += nt) {
      const int pj = parent ? parent[row + j] : j - 1;
      s_par[j] = pj;
      s_pos[j] = -1;
      s_acc[j + 1] = n;  // no accepted child
      if (pj < -1 || pj >= j) local_bad = 1;
    }
    if (tid == 0) s_acc[0] = n;
    // barrier + block-wide OR: every thread gets the same verdict
    bool bad = __syncthreads_or(local_bad) != 0;
    if (!bad) {
      // the path: node i is a child of node i - 1 (the root for i = 0)
      int path_bad = 0;
      for (int i = tid; i < len; i += nt) {
        const int v = path ? path[row + i] : i;
        const int prev = i ? (path ? path[row + i - 1] : i - 1) : -1;
        if (v < 0 || v >= n || prev < -1 || prev >= n || s_par[v] != prev) {
          path_bad = 1;
        } else {
          s_pos[v] = i;
          s_acc[prev + 1] = v;
        }
      }
      bad = __syncthreads_or(path_bad) != 0;
    }
    if (!bad) {
      for (int j = tid; j < n; j += nt) {
        const int pj = s_par[j];
        const int ppos = pj < 0 ? -1 : s_pos[pj];
        if ((pj < 0 || ppos >= 0) && j <= s_acc[pj + 1])
          C.add(j, ppos + 2, s_pos[j] >= 0, C.calib ? conf[row + j] : 0.f);
      }
    }
    if (tid == 0) atomicAdd(bad ? C.inv : &C.len[len], 1u);
    __syncthreads();
  }
  C.flush(out, n);
}

template <typename K>
cudaError_t launch(K kernel, int grid, int threads, size_t smem, cudaStream_t st,
                   const int32_t* count, const int32_t* parent, const int32_t* path,
                   const float* conf, int B, const StatsSmem& L, const spec_accept_stats_t& out) {
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  prof_begin(SPEC_PROF_STATS, st);
  kernel<<<grid, threads, smem, st>>>(count, parent, path, conf, B, L, out);
  prof_end(SPEC_PROF_STATS, st);
  return cudaGetLastError();
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" int spec_accept_stats(const int32_t* count, const int32_t* parent,
                                 const int32_t* path_nodes, const float* confidence, int B, int n,
                                 int nbins, const spec_accept_stats_t* out, void* stream) {
  if (!out || !count) return SPEC_ERR_ARG;
  if (B < 0 || n < 1 || n > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  const bool tree = parent != nullptr;
  if (tree != (path_nodes != nullptr)) return SPEC_ERR_ARG;
  const bool calib = confidence != nullptr;
  if (calib && (nbins < 1 || nbins > SPEC_STATS_MAX_BINS)) return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  // element alignment of every array (a misaligned pointer is an argument
  // error here, not a fault on the device)
  const uintptr_t a4 = (uintptr_t)count | (uintptr_t)parent | (uintptr_t)path_nodes |
                       (uintptr_t)confidence;
  const uintptr_t a8 = (uintptr_t)out->len_hist | (uintptr_t)out->node_tested |
                       (uintptr_t)out->node_accepted | (uintptr_t)out->depth_tested |
                       (uintptr_t)out->depth_accepted | (uintptr_t)out->calib_tested |
                       (uintptr_t)out->calib_accepted | (uintptr_t)out->calib_conf_sum |
                       (uintptr_t)out->invalid;
  if (a4 % 4 != 0 || a8 % 8 != 0) return SPEC_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (n <= kWarpNodes) {
    const StatsSmem L = plan(n, calib ? nbins : 0, tree, calib, true);
    // up to eight 256-thread CTAs per SM (full occupancy); beyond that
    // each warp takes several rounds, which bounds the flush's atomics
    const int64_t want = ((int64_t)B + kStatsWarps - 1) / kStatsWarps;
    const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);
    e = tree ? launch(accept_stats_warp<true>, grid, kStatsWarps * 32, L.bytes(), st, count,
                      parent, path_nodes, confidence, B, L, *out)
             : launch(accept_stats_warp<false>, grid, kStatsWarps * 32, L.bytes(), st, count,
                      nullptr, nullptr, confidence, B, L, *out);
  } else {
    const StatsSmem L = plan(n, calib ? nbins : 0, true, calib, false);
    const int grid = B < 2 * sms ? B : 2 * sms;
    e = launch(accept_stats_cta, grid, 256, L.bytes(), st, count, parent, path_nodes,
               confidence, B, L, *out);
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
