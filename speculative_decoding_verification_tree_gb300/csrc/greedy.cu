// Greedy (temperature 0) verification: "贪婪情形简化" of "投机解码与 EAGLE" --
// accept while the drafted token equals argmax of the target logits at its
// position, then emit that argmax.  For trees the accepted child of a row is
// the first child (index order) whose token is the row's argmax.
//
// Two kernels.  argmax_partial streams every target row once (HBM bound:
// 2 or 4 bytes per logit, nothing else read) and reduces chunks of
// kArgChunk logits to (value, lowest index) pairs; greedy_finalize reduces
// each row's chunk results, walks each sequence and writes the outputs.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// (v, i) beats (bv, bi): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void consider(float raw, int idx, float& bv, int& bi) {
  const float v = fmaxf(raw, neg_inf());  // NaN reads as -inf
  if (v > bv) {
    bv = v;
    bi = idx;
  }
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads) argmax_partial(const T* __restrict__ x, int V, int S,
                                                           ArgPart* __restrict__ part) {
  launch_dependents();  // greedy_finalize waits for this grid itself
  const int64_t item = blockIdx.x;
  const int64_t row = item / S;
  const int s = (int)(item - row * S);
  const T* rp = x + row * (int64_t)V;
  const int c0 = s * kArgChunk;
  const int c1 = min(V, c0 + kArgChunk);
  float bv = neg_inf();
  int bi = INT_MAX;
  if constexpr (kVec) {
    constexpr int kEpv = 16 / (int)sizeof(T);            // elements per 16-byte vector
    constexpr int kNv = kArgChunk / kEpv / kThreads;      // vectors per thread
    uint4 buf[kNv];
    const int first = c0 + threadIdx.x * kEpv;
    if (first < c1) bi = first;  // all -inf: lowest index this thread sees
#pragma unroll
    for (int j = 0; j < kNv; ++j) {
      const int e = c0 + (threadIdx.x + kThreads * j) * kEpv;
      if (e < c1) buf[j] = ldg_stream(rp + e);
    }
#pragma unroll
    for (int j = 0; j < kNv; ++j) {
      const int e = c0 + (threadIdx.x + kThreads * j) * kEpv;
      if (e < c1) {
        if constexpr (sizeof(T) == 2) {
          const uint32_t w[4] = {buf[j].x, buf[j].y, buf[j].z, buf[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            consider(bf16_lo(w[q]), e + 2 * q, bv, bi);
            consider(bf16_hi(w[q]), e + 2 * q + 1, bv, bi);
          }
        } else {
          consider(__uint_as_float(buf[j].x), e, bv, bi);
          consider(__uint_as_float(buf[j].y), e + 1, bv, bi);
          consider(__uint_as_float(buf[j].z), e + 2, bv, bi);
          consider(__uint_as_float(buf[j].w), e + 3, bv, bi);
        }
      }
    }
  } else {
    if (c0 + (int)threadIdx.x < c1) bi = c0 + threadIdx.x;
    for (int e = c0 + threadIdx.x; e < c1; e += kThreads) consider(ElemIO<T>::get(rp, e), e, bv, bi);
  }
  // warp then block reduction under the tie rule
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  __shared__ float sv_[kThreads / 32];
  __shared__ int si_[kThreads / 32];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sv_[w] = bv;
    si_[w] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kThreads / 32; ++k)
      if (better(sv_[k], si_[k], bv, bi)) {
        bv = sv_[k];
        bi = si_[k];
      }
    part[item] = ArgPart{bv, bi};
  }
}

// One CTA per sequence: row argmaxes, first matching child per row, walk.
__global__ void __launch_bounds__(kThreads) greedy_finalize(VerifyShape s, VerifyArgs a, int S) {
  extern __shared__ int32_t sh[];
  // a programmatic dependent of argmax_partial: nothing read before it is done
  grid_dependency_wait();
  const int n = s.n;
  int32_t* g = sh;               // [n+1] argmax per row
  int32_t* first = sh + n + 1;   // [n+1] first matching child
  int32_t* haskid = first + n + 1;
  __shared__ int s_len;
  const int b = blockIdx.x;
  const int64_t row0 = (int64_t)b * (n + 1);
  for (int r = threadIdx.x; r <= n; r += blockDim.x) {
    const ArgPart* pp = a.arg_part + (row0 + r) * S;
    float bv = pp[0].v;
    int bi = pp[0].i;
    for (int k = 1; k < S; ++k)
      if (better(pp[k].v, pp[k].i, bv, bi)) {
        bv = pp[k].v;
        bi = pp[k].i;
      }
    g[r] = (bi == INT_MAX) ? 0 : bi;
    first[r] = INT_MAX;
    haskid[r] = 0;
  }
  __syncthreads();
  const int32_t* toks = a.node_tokens + (int64_t)b * n;
  uint32_t bad = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int p = s.chain ? j - 1 : a.parent[(int64_t)b * n + j];
    if (p < -1 || p >= j) {
      bad |= SPEC_STATUS_BAD_TREE;
      continue;
    }
    const int r = p + 1;
    haskid[r] = 1;
    const int t = toks[j];
    if (t < 0 || t >= s.V) bad |= SPEC_STATUS_TOKEN_RANGE;
    if (t == g[r]) atomicMin(&first[r], j);
  }
  if (bad) flag_status(a.status, bad);
  __syncthreads();
  // acceptance mass of point-mass distributions
  for (int r = threadIdx.x; r <= n; r += blockDim.x) {
    if (s.chain) {
      if (r < n) a.mass[(int64_t)b * n + r] = (toks[r] == g[r]) ? 1.f : 0.f;
    } else {
      a.mass[row0 + r] = haskid[r] ? (first[r] != INT_MAX ? 1.f : 0.f) : __int_as_float(0x7fc00000);
    }
  }
  int32_t* out = a.out_tokens + (int64_t)b * (n + 1);
  if (threadIdx.x == 0) {
    int r = 0, len = 0;
    while (first[r] != INT_MAX) {
      const int j = first[r];
      if (!s.chain) a.path_nodes[(int64_t)b * n + len] = j;
      out[len] = toks[j];
      ++len;
      r = j + 1;
    }
    out[len] = g[r];
    a.count[b] = len;
    s_len = len;
  }
  __syncthreads();
  const int len = s_len;
  for (int k = len + 1 + threadIdx.x; k <= n; k += blockDim.x) out[k] = -1;
  if (!s.chain)
    for (int k = len + threadIdx.x; k < n; k += blockDim.x) a.path_nodes[(int64_t)b * n + k] = -1;
}

}  // namespace

cudaError_t launch_greedy(const VerifyShape& s, const VerifyArgs& a, cudaStream_t st) {
  const int S = arg_splits(s.V);
  const int64_t items = s.rows() * S;
  const size_t esz = a.dt_target == SPEC_BF16 ? 2 : 4;
  const bool vec = ((uintptr_t)a.target % 16 == 0) && ((s.V * esz) % 16 == 0);
  if (items > 0) {
    prof_begin(SPEC_PROF_ARGMAX, st);
    if (a.dt_target == SPEC_BF16) {
      const uint16_t* t = (const uint16_t*)a.target;
      if (vec)
        argmax_partial<uint16_t, true><<<(unsigned)items, kThreads, 0, st>>>(t, s.V, S, a.arg_part);
      else
        argmax_partial<uint16_t, false><<<(unsigned)items, kThreads, 0, st>>>(t, s.V, S, a.arg_part);
    } else {
      const float* t = (const float*)a.target;
      if (vec)
        argmax_partial<float, true><<<(unsigned)items, kThreads, 0, st>>>(t, s.V, S, a.arg_part);
      else
        argmax_partial<float, false><<<(unsigned)items, kThreads, 0, st>>>(t, s.V, S, a.arg_part);
    }
    cudaError_t e = cudaGetLastError();
    prof_end(SPEC_PROF_ARGMAX, st);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = (size_t)3 * (s.n + 1) * sizeof(int32_t);
  // a programmatic dependent launch: its CTAs take the SMs the partial
  // argmax leaves and start the moment that grid completes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, greedy_finalize, s, a, S);
}

}  // namespace sv
