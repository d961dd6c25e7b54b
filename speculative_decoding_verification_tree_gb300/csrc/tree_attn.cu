// spec_tree_attention: attention of the verification pass over a draft tree.
//
// EAGLE-2 notes §4.2: the selected draft tokens are flattened into one
// sequence and verified in one forward pass; each drafted token may see the
// committed prefix, its ancestors and itself, never another branch.  For
// sequence b with prefix length P (keys / values at cache positions
// 0 .. P-1) and drafted node i (key / value at position P + i):
//
//   o_i = softmax over visible keys s of (scale * q_i . k_s), applied to v_s,
//   visible = {0 .. P-1} + {P + j : bit j of mask_bits[b, i]}
//
// with grouped-query heads (query head h reads key/value head h / (Hq/Hkv)).
//
// Organisation (head dim 128, bf16, fp32 accumulation).  A CTA takes 64 query
// rows of one (sequence, key/value head): the rows are (node, head in the
// group) pairs, node-major, so the G query heads that share a key/value head
// are served by one read of its keys and values.  Four warps of 16 rows each
// run the FlashAttention-2 recurrence on tensor cores (mma.sync m16n8k16
// bf16): S = Q K^T per 64-key tile from a double-buffered cp.async ring in
// shared memory (K fragments by ldmatrix, V fragments by ldmatrix.trans), the
// tree mask applied only in tiles that reach the drafted positions, an
// online base-2 softmax in registers, and P V accumulated in registers.
#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kAD = 128;            // head dim
constexpr int kAKeys = 64;          // keys per tile
constexpr int kARows = 64;          // query rows per CTA (4 warps x 16)
constexpr int kAThreads = 128;
constexpr int kAPitch = kAD + 8;    // smem row pitch in bf16 (272 bytes: no bank conflicts)
constexpr int kATile = kAKeys * kAPitch;  // bf16 elements per tile buffer

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two floats -> bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kAThreads, 3)
    tree_attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kc,
                     const uint16_t* __restrict__ vc, const int32_t* __restrict__ prefix_len,
                     const uint64_t* __restrict__ mask_bits, int N, int Hq, int Hkv, int S,
                     float scale_log2, uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) uint16_t asmem[];
  uint16_t* Ks = asmem;                // [2][64][kAPitch]
  uint16_t* Vs = asmem + 2 * kATile;   // [2][64][kAPitch]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int G = Hq / Hkv, R = N * G;

  int P = prefix_len[b];
  P = P < 0 ? 0 : (P > S - N ? S - N : P);
  const int L = P + N;  // keys of this sequence
  const int64_t kvbase = ((int64_t)b * Hkv + kvh) * S * kAD;

  // this thread's two rows (g and g + 8 of the warp's 16)
  int node[2], hq[2];
  bool valid[2];
  uint64_t mb[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = blockIdx.x * kARows + warp * 16 + g + 8 * h;
    valid[h] = r < R;
    node[h] = valid[h] ? r / G : 0;
    hq[h] = kvh * G + (valid[h] ? r % G : 0);
    mb[h] = valid[h] ? mask_bits[(int64_t)b * N + node[h]] : ~0ull;
  }
  // Q fragments (A operand), 8 k-steps of 16 over the head dim
  uint32_t qf[8][4];
  {
    const uint32_t* q0 =
        reinterpret_cast<const uint32_t*>(q + (((int64_t)b * N + node[0]) * Hq + hq[0]) * kAD);
    const uint32_t* q1 =
        reinterpret_cast<const uint32_t*>(q + (((int64_t)b * N + node[1]) * Hq + hq[1]) * kAD);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c = kk * 8 + t4;  // 32-bit word: elements kk*16 + 2 t4, +1
      qf[kk][0] = valid[0] ? q0[c] : 0u;
      qf[kk][1] = valid[1] ? q1[c] : 0u;
      qf[kk][2] = valid[0] ? q0[c + 4] : 0u;
      qf[kk][3] = valid[1] ? q1[c + 4] : 0u;
    }
  }

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {neg_inf(), neg_inf()}, l[2] = {0.f, 0.f};

  // one tile of keys and values into buffer `buf` (keys past L are zeros)
  auto load_tile = [&](int tile, int buf) {
    const uint32_t kd = smem_u32(Ks + buf * kATile), vd = smem_u32(Vs + buf * kATile);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = tid + i * kAThreads;  // 16-byte chunk: key c / 16, column (c % 16) * 8
      const int kr = c >> 4, col = (c & 15) * 8;
      const int key = tile * kAKeys + kr;
      const bool ok = key < L;
      const int64_t src = kvbase + (int64_t)(ok ? key : 0) * kAD + col;
      const uint32_t off = (uint32_t)((kr * kAPitch + col) * 2);
      cp_async16(kd + off, kc + src, ok ? 16u : 0u);
      cp_async16(vd + off, vc + src, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  const int ntile = (L + kAKeys - 1) / kAKeys;
  load_tile(0, 0);
  for (int tile = 0; tile < ntile; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < ntile) {
      load_tile(tile + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kb = smem_u32(Ks + buf * kATile), vb = smem_u32(Vs + buf * kATile);

    // S = Q K^T for 64 keys: 8 key groups of 8 (n) x 8 head-dim steps (k)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        // matrices: (keys 8j.., dims 32 k2 + 8 mi), mi = lane / 8
        const uint32_t addr =
            kb + (uint32_t)(((j * 8 + (lane & 7)) * kAPitch + k2 * 32 + (lane >> 3) * 8) * 2);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma_bf16(s[j], qf[2 * k2], b0, b1);
        mma_bf16(s[j], qf[2 * k2 + 1], b2, b3);
      }
    }
    // scale to base 2; mask where the tile reaches the drafted positions
    const int key0 = tile * kAKeys;
    const bool masked = key0 + kAKeys > P;
    float mx[2] = {neg_inf(), neg_inf()};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        float v = s[j][e] * scale_log2;
        if (masked) {
          const int key = key0 + j * 8 + 2 * t4 + (e & 1);
          const int tj = key - P;
          const bool vis = key < P || (tj < N && ((mb[h] >> tj) & 1ull));
          if (!vis) v = neg_inf();
        }
        s[j][e] = v;
        mx[h] = fmaxf(mx[h], v);
      }
    }
    float corr[2], mu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mn = fmaxf(m[h], mx[h]);
      mu[h] = mn == neg_inf() ? 0.f : mn;  // no visible key yet: nothing to scale
      corr[h] = ex2(m[h] - mu[h]);
      m[h] = mn;
      l[h] *= corr[h];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    // P = 2^(s - m) as bf16 A fragments, 4 steps of 16 keys
    uint32_t pf[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float p[2][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = 2 * kk + hh;
        p[hh][0] = ex2(s[j][0] - mu[0]);
        p[hh][1] = ex2(s[j][1] - mu[0]);
        p[hh][2] = ex2(s[j][2] - mu[1]);
        p[hh][3] = ex2(s[j][3] - mu[1]);
        l[0] += p[hh][0] + p[hh][1];
        l[1] += p[hh][2] + p[hh][3];
      }
      pf[kk][0] = pack_bf16(p[0][0], p[0][1]);
      pf[kk][1] = pack_bf16(p[0][2], p[0][3]);
      pf[kk][2] = pack_bf16(p[1][0], p[1][1]);
      pf[kk][3] = pack_bf16(p[1][2], p[1][3]);
    }
    // O += P V: 16 head-dim groups of 8 (n) x 4 key steps of 16 (k)
#pragma unroll
    for (int jd = 0; jd < 16; jd += 2) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // matrices: (keys 16 kk + 8 (mi & 1), dims 8 jd + 8 (mi >> 1)), mi = lane / 8
        const int mi = lane >> 3;
        const uint32_t addr = vb + (uint32_t)(((kk * 16 + (mi & 1) * 8 + (lane & 7)) * kAPitch +
                                               jd * 8 + (mi >> 1) * 8) * 2);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma_bf16(o[jd], pf[kk], b0, b1);
        mma_bf16(o[jd + 1], pf[kk], b2, b3);
      }
    }
    __syncthreads();  // the buffer is refilled by the next iteration's load
  }

  // normalise and store: rows g (c0, c1) and g + 8 (c2, c3)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
  const float inv0 = 1.f / l[0], inv1 = 1.f / l[1];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!valid[h]) continue;
    uint32_t* dst =
        reinterpret_cast<uint32_t*>(out + (((int64_t)b * N + node[h]) * Hq + hq[h]) * kAD);
    const float inv = h ? inv1 : inv0;
#pragma unroll
    for (int jd = 0; jd < 16; ++jd)
      dst[jd * 4 + t4] = pack_bf16(o[jd][2 * h] * inv, o[jd][2 * h + 1] * inv);
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" int spec_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* prefix_len, const uint64_t* mask_bits, int B,
                                   int N, int Hq, int Hkv, int D, int S, float scale, void* out,
                                   void* stream) {
  // B and Hkv index grid dimensions z and y (at most 65535 each)
  if (B < 0 || B > 65535 || N < 1 || N > 64 || Hq < 1 || Hkv < 1 || Hkv > 65535 ||
      Hq % Hkv != 0 || S < N)
    return SPEC_ERR_SHAPE;
  if (D != kAD) return SPEC_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < 3.4e38f)) return SPEC_ERR_ARG;
  if (B == 0) return SPEC_OK;
  if (!q || !k_cache || !v_cache || !prefix_len || !mask_bits || !out) return SPEC_ERR_ARG;
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0 ||
      ((uintptr_t)q | (uintptr_t)out | (uintptr_t)prefix_len) % 4 != 0 ||
      (uintptr_t)mask_bits % 8 != 0)
    return SPEC_ERR_ARG;
  const int R = N * (Hq / Hkv);
  const dim3 grid((unsigned)((R + kARows - 1) / kARows), (unsigned)Hkv, (unsigned)B);
  const size_t smem = (size_t)4 * kATile * sizeof(uint16_t);
  if (cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  prof_begin(SPEC_PROF_ATTN, st);
  tree_attn_kernel<<<grid, kAThreads, smem, st>>>(
      (const uint16_t*)q, (const uint16_t*)k_cache, (const uint16_t*)v_cache, prefix_len,
      mask_bits, N, Hq, Hkv, S, scale * kLog2e, (uint16_t*)out);
  prof_end(SPEC_PROF_ATTN, st);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
