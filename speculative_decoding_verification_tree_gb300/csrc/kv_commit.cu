// spec_kv_commit: keep the accepted drafts' KV entries after verification
// ("KV cache rollback" of the Vietnamese speculative-decoding page; "El baile
// de caché KV" of the Spanish page).
//
// A chain only sets the logical lengths.  A tree moves the accepted path's
// entries (node order after the prefix) to consecutive positions in path
// order.  Each thread owns one word of one row of one plane of one sequence,
// so no two threads touch the same bytes.  The path's nodes increase and
// node_i >= i, so no source node_k is the destination j < k of an earlier
// step: a thread may read the sources of up to kBatch path positions into
// registers and then store them all (one memory round trip per batch rather
// than per position).  Pure data movement: HBM-bound, algorithmic bytes =
// 2 x row_bytes x planes per moved position.
#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kKvThreads = 256;
constexpr int kBatch = 8;  // path positions whose sources are read before any store

// Runs after kv_lengths: new_len[b] = prefix[b] + path length for a valid
// path, -1 otherwise (then nothing moves).
template <typename W>
__global__ void __launch_bounds__(kKvThreads) kv_move(unsigned char* __restrict__ kv, int B, int n1,
                                                      int n2, int64_t sb, int64_t s1, int64_t s2,
                                                      int64_t sp, int words,
                                                      const int32_t* __restrict__ prefix,
                                                      const int32_t* __restrict__ nodes,
                                                      const int32_t* __restrict__ new_len, int N) {
  // work item = (b, p1, p2, word), word fastest
  const int64_t per_b = (int64_t)n1 * n2 * words;
  const int64_t total = (int64_t)B * per_b;
  for (int64_t t = blockIdx.x * (int64_t)kKvThreads + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * kKvThreads) {
    const int b = (int)(t / per_b);
    int64_t r = t - (int64_t)b * per_b;
    const int w = (int)(r % words);
    r /= words;
    const int p2 = (int)(r % n2);
    const int p1 = (int)(r / n2);
    const int32_t* nb = nodes + (int64_t)b * N;
    const int nl = new_len[b], pre = prefix[b];
    if (nl < 0) continue;  // invalid path
    const int len = nl - pre;
    unsigned char* base = kv + (int64_t)b * sb + (int64_t)p1 * s1 + (int64_t)p2 * s2 +
                          (int64_t)pre * sp + (int64_t)w * sizeof(W);
    for (int i0 = 0; i0 < len; i0 += kBatch) {
      W v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k;
        if (i < len && nb[i] != i) v[k] = *reinterpret_cast<const W*>(base + (int64_t)nb[i] * sp);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k;
        if (i < len && nb[i] != i) *reinterpret_cast<W*>(base + (int64_t)i * sp) = v[k];
      }
    }
  }
}

// One warp per sequence: the lanes load 32 path nodes at a time and test
// them together (each above its predecessor, below N).
__global__ void kv_lengths(int B, const int32_t* __restrict__ prefix,
                           const int32_t* __restrict__ nodes, const int32_t* __restrict__ plen,
                           int N, int32_t* __restrict__ new_len) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (b >= B) return;  // whole warps leave together
  const int len = plen[b];
  bool ok = len >= 0 && len <= N;
  if (ok && nodes) {
    const int32_t* nb = nodes + (int64_t)b * N;
    int carry = -1;  // the node before this group of 32
    for (int i0 = 0; i0 < len; i0 += 32) {
      const int i = i0 + lane;
      const int v = i < len ? nb[i] : 0;
      int prev = __shfl_up_sync(0xffffffffu, v, 1);
      if (lane == 0) prev = carry;
      const bool bad = i < len && (v <= prev || v >= N);
      if (__any_sync(0xffffffffu, bad)) {
        ok = false;
        break;
      }
      carry = __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (lane == 0) new_len[b] = ok ? prefix[b] + len : -1;
}

template <typename W>
cudaError_t launch_move(unsigned char* kv, int B, int n1, int n2, int64_t sb, int64_t s1,
                        int64_t s2, int64_t sp, int row_bytes, const int32_t* prefix,
                        const int32_t* nodes, const int32_t* new_len, int N, cudaStream_t st) {
  const int words = row_bytes / (int)sizeof(W);
  const int64_t total = (int64_t)B * n1 * n2 * words;
  if (total == 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  if (e != cudaSuccess) return e;
  const int64_t want = (total + kKvThreads - 1) / kKvThreads;
  const int64_t cap = (int64_t)sms * 8;  // eight 256-thread CTAs per SM
  prof_begin(SPEC_PROF_KV, st);
  kv_move<W><<<(unsigned)(want < cap ? want : cap), kKvThreads, 0, st>>>(
      kv, B, n1, n2, sb, s1, s2, sp, words, prefix, nodes, new_len, N);
  prof_end(SPEC_PROF_KV, st);
  return cudaGetLastError();
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" int spec_kv_commit(void* kv, int B, int n1, int n2, int64_t stride_b,
                              int64_t stride_1, int64_t stride_2, int64_t stride_pos,
                              int row_bytes, const int32_t* prefix_len,
                              const int32_t* path_nodes, const int32_t* path_len, int N,
                              int32_t* new_len, void* stream) {
  if (B < 0 || n1 < 0 || n2 < 0 || N < 0 || row_bytes < 0) return SPEC_ERR_SHAPE;
  if (stride_b < 0 || stride_1 < 0 || stride_2 < 0 || stride_pos < 0) return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  if (!prefix_len || !path_len || !new_len) return SPEC_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const bool moves = path_nodes && n1 > 0 && n2 > 0 && row_bytes > 0;
  if (moves && !kv) return SPEC_ERR_ARG;
  // lengths first: they validate each path once for the move kernel
  kv_lengths<<<(B + 7) / 8, 256, 0, st>>>(B, prefix_len, path_nodes, path_len, N, new_len);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (moves) {
    unsigned char* p = (unsigned char*)kv;
    // widest word that every address of the layout is aligned to
    uint64_t g = (uint64_t)(uintptr_t)p | (uint64_t)row_bytes | (uint64_t)stride_b |
                 (uint64_t)stride_1 | (uint64_t)stride_2 | (uint64_t)stride_pos;
    cudaError_t e;
    if (g % 16 == 0)
      e = launch_move<uint4>(p, B, n1, n2, stride_b, stride_1, stride_2, stride_pos, row_bytes,
                             prefix_len, path_nodes, new_len, N, st);
    else if (g % 4 == 0)
      e = launch_move<uint32_t>(p, B, n1, n2, stride_b, stride_1, stride_2, stride_pos, row_bytes,
                                prefix_len, path_nodes, new_len, N, st);
    else
      e = launch_move<unsigned char>(p, B, n1, n2, stride_b, stride_1, stride_2, stride_pos,
                                     row_bytes, prefix_len, path_nodes, new_len, N, st);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}
