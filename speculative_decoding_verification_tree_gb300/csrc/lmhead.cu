// Target LM head of the verification pass on the fifth-generation tensor
// cores (tcgen05 + TMEM + TMA), with the first pass of verification in the
// epilogue.
//
// Step 2 of the draft/verify loop ("投机解码与 EAGLE", the four steps of one
// round) runs the target once over every drafted position; its last layer
// maps each position's final hidden state h [H] to logits over the
// vocabulary, z = W h with W [V, H] (the LM head).  Here that product is one
// GEMM, logits [M, V] = hidden [M, H] x W^T, accumulated in float32 in TMEM,
// rounded to bf16 (the logits a bf16 forward pass produces) and written out.
// The epilogue also takes the first verification pass over the tile it holds:
// the base-2 maximum and sum of 2^(z kt - max), kt = log2(e) / T, over each
// row's 256 columns, so that verification needs no separate pass to find the
// target rows' normalisers.
//
// Kernel shape (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0     TMA producer: 128-byte-swizzled K-major tiles of hidden
//              (128 x 64) and W (256 x 64) into a 4-stage shared-memory ring;
//   warp 1     allocates 512 TMEM columns (two 128 x 256 float32
//              accumulators) and issues tcgen05.mma (M 128, N 256, K 16, bf16
//              in, float32 out) from one thread; tcgen05.commit frees ring
//              stages and hands finished accumulators to the epilogue;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//              row per thread), bf16 rounding, stores, tile statistics.
// Tiles are taken in vocabulary-block-major order so that the CTAs working at
// one time share a few 256-row slices of W through L2 while the hidden states
// (a few MB) stay resident.  CTAs run in clusters of two that take the two
// 128-row halves of a 256-row block of the same W tile: each loads its own
// hidden tile and one 128-row half of the W tile, multicast into both CTAs'
// shared memory, so a CTA pulls 32 KB instead of 48 KB from L2 per K step; a
// ring stage is refilled only when both CTAs' MMAs have released it (each
// MMA commit arrives on both CTAs' "empty" barriers).  Every mbarrier wait is bounded: a wait that gives
// up sets SPEC_STATUS_TIMEOUT and a CTA-wide flag after which no wait blocks,
// and before TMEM is freed the CTA waits (again bounded) for its own MMAs and
// copies in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTmemCols = 2 * BN;  // two float32 accumulators
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;

struct __align__(8) GemmSmem {
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[2], tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t dead;
};
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 + sizeof(GemmSmem);

struct GemmParams {
  int M, N, K;
  int nm, nn, ntiles, nkb;  // ntiles: work units (tiles, or tile pairs)
  uint16_t* logits;  // [M, ldo] bf16 bits
  int64_t ldo;
  float2* stats;     // [M, nn] (max, sum) in base 2 at kt, or null
  float kt;
  uint32_t* status;
  int test_stall;  // withhold the first stage's copies (bounded-wait test)
};

// Bounded wait on a CTA barrier that gives up at once when the CTA is dead.
__device__ __forceinline__ void gwait(GemmSmem& sm, uint64_t* bar, uint32_t parity,
                                      uint32_t* status) {
  if (*(volatile uint32_t*)&sm.dead) return;
  if (!mbar_wait_bounded(bar, parity)) {
    *(volatile uint32_t*)&sm.dead = 1;
    flag_status(status, SPEC_STATUS_TIMEOUT);
  }
}

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 64 bf16 (128 B), 8-row groups 1024 B apart; the tile starts on a
// 1024-byte boundary so the base offset is 0.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride between 8-row groups
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), float32 D,
// M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4)            // D float32
                            | (1u << 7)          // A bf16
                            | (1u << 10)         // B bf16
                            | ((uint32_t)(BN >> 3) << 17)
                            | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The same box into this CTA and its cluster peer (same shared-memory
// offsets), completing its bytes on each CTA's barrier at `bar`'s offset.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint64_t* bar, uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster.L2::cache_hint [%0], [%1, {%4, %5}], [%2], %3, %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "h"(mask), "r"(x), "r"(y),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Commit arriving on the barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// 32 consecutive float32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int CL>  // CTAs per cluster: 1, or 2 sharing each W tile
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                GemmParams P) {
  const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
  const int unit0 = CL == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = CL == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int nmu = CL == 2 ? (P.nm + 1) >> 1 : P.nm;  // M units per W tile
  // work unit -> (m tile, n tile) of this CTA
  auto tile_of = [&](int t, int& mb, int& nb) {
    nb = t / nmu;
    mb = CL == 2 ? 2 * (t - nb * nmu) + rank : t - nb * nmu;
  };
  extern __shared__ __align__(1024) unsigned char dyn_raw[];
  // the ring starts on a 1024-byte boundary (128-byte swizzle atoms)
  const uint32_t raw = smem_u32(dyn_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  unsigned char* ring_ptr = dyn_raw + (ring - raw);
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(ring_ptr + (size_t)kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CL);  // released by the MMAs of every CTA
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.tfull[a], 1);
      mbar_init(&sm.tempty[a], kEpiThreads);
    }
    mbar_init(&sm.drain, 1);
    sm.dead = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (CL == 2) cluster_sync();  // the peer's barriers exist before any multicast
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint64_t pol_a, pol_b;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_a));
      asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_b));
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fills[kStages] = {};  // copies issued into each stage
      bool stall_pending = blockIdx.x == 0;  // the test stall: CTA 0 only
      for (int t = unit0; t < P.ntiles; t += units) {
        int mb, nb;
        tile_of(t, mb, nb);
        for (int kb = 0; kb < P.nkb; ++kb) {
          gwait(sm, &sm.empty[stage], phase ^ 1u, P.status);
          const uint32_t sa = ring + (uint32_t)(stage * kStageBytes);
          if (P.test_stall && stall_pending) {
            // test only: this stage is never filled; the MMA issuer's wait on
            // it gives up and the CTA finishes without waiting any further
            stall_pending = false;
          } else {
            mbar_expect_tx(&sm.full[stage], (uint32_t)kStageBytes);
            tma_load_2d(sa, &map_a, kb * BK, mb * BM, &sm.full[stage], pol_a);
            if constexpr (CL == 2) {
              // this CTA's half of the W tile, into both CTAs
              const uint32_t half = (uint32_t)(kBBytes / 2);
              tma_load_2d_mc(sa + kABytes + (uint32_t)rank * half, &map_b, kb * BK,
                             nb * BN + rank * (BN / 2), &sm.full[stage], (uint16_t)3, pol_b);
            } else {
              tma_load_2d(sa + kABytes, &map_b, kb * BK, nb * BN, &sm.full[stage], pol_b);
            }
            ++fills[stage];
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // wait for this CTA's last copy into each stage (normally consumed
      // already; after a timeout they may still be in flight)
      for (int s = 0; s < kStages; ++s)
        if (fills[s] > 0) mbar_wait_bounded(&sm.full[s], (fills[s] - 1) & 1u);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int t = unit0; t < P.ntiles; t += units) {
        gwait(sm, &sm.tempty[acc], acc_phase ^ 1u, P.status);
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < P.nkb; ++kb) {
          gwait(sm, &sm.full[stage], phase, P.status);
          tc_fence_after();
          const uint32_t sa = ring + (uint32_t)(stage * kStageBytes);
          const uint64_t da = sw128_desc(sa), db = sw128_desc(sa + kABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // +32 bytes of K per step
            umma_bf16(d, da + 2u * k, db + 2u * k, (kb | k) != 0 ? 1u : 0u);
          if constexpr (CL == 2) umma_commit_mc(&sm.empty[stage], (uint16_t)3);
          else umma_commit(&sm.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(&sm.tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA this thread issued has completed before TMEM is freed
      umma_commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    const bool vec = (P.ldo % 8) == 0 && ((uintptr_t)P.logits % 16) == 0;
    for (int t = unit0; t < P.ntiles; t += units) {
      int mb, nb;
      tile_of(t, mb, nb);
      gwait(sm, &sm.tfull[acc], acc_phase, P.status);
      tc_fence_after();
      const int row = mb * BM + r_in;
      const bool live = row < P.M;  // (the odd last M tile's partner: none)
      uint16_t* out = P.logits + (int64_t)(live ? row : 0) * P.ldo;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      float m = neg_inf(), s = 0.f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int col0 = nb * BN + c * 32;
        if (col0 >= P.N) break;  // the same for every thread of the warp
        uint32_t r[32];
        tmem_ld32(tbase + (uint32_t)(c * 32), r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 h =
              __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          pk[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const int nval = min(32, P.N - col0);
        if (P.stats) {
          float x[32];
          float mc = neg_inf();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            x[2 * i] = bf16_lo(pk[i]) * P.kt;
            x[2 * i + 1] = bf16_hi(pk[i]) * P.kt;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i >= nval) x[i] = neg_inf();
            mc = fmaxf(mc, x[i]);
          }
          if (mc > m) {
            s = (m == neg_inf()) ? 0.f : s * ex2(m - mc);
            m = mc;
          }
          float acc_s = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) acc_s += ex2(x[i] - m);
          s += acc_s;
        }
        if (live) {
          if (vec && nval == 32) {
            uint4* dst = reinterpret_cast<uint4*>(out + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)  // constant indices keep pk in registers
              if (i < nval)
                out[col0 + i] = (uint16_t)((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xffffu));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.tempty[acc]);
      if (P.stats && live) P.stats[(int64_t)row * P.nn + nb] = make_float2(m, s);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer may still multicast into it or arrive on
  // its barriers
  if (CL == 2) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// Per row: combine the tile statistics into the row's base-2 log normaliser
// L = max + log2(sum) (one warp per row).
__global__ void lse_merge(const float2* __restrict__ stats, int M, int nn, float* __restrict__ lse) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  MaxSum a{neg_inf(), 0.f};
  for (int i = lane; i < nn; i += 32) {
    const float2 v = stats[(int64_t)row * nn + i];
    a = ms_combine(a, MaxSum{v.x, v.y});
  }
  a = warp_ms(a);
  if (lane == 0) lse[row] = a.m + log2f(a.z);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, K] bf16 matrix as K-major 64 x box_rows tiles, 128-byte
// swizzle, zero fill outside.
bool make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int lmhead_tiles_n(int V) { return (V + BN - 1) / BN; }

bool lmhead_supported(const void* hidden, const void* w, int H) {
  return H >= 8 && H % 8 == 0 && (uintptr_t)hidden % 16 == 0 && (uintptr_t)w % 16 == 0;
}

cudaError_t launch_lmhead(const void* hidden, const void* w, int M, int H, int V, float temperature,
                          uint16_t* logits, int64_t ldo, float2* stats, float* lse,
                          uint32_t* status, cudaStream_t st, bool test_stall) {
  if (M == 0) return cudaSuccess;
  if (!lmhead_supported(hidden, w, H)) return cudaErrorInvalidValue;
  // clusters of two CTAs share each W tile when there are two M tiles to pair
  const int nm = (M + BM - 1) / BM;
  const int CL = nm >= 2 ? 2 : 1;
  CUtensorMap ma, mb;
  if (!make_map(&ma, hidden, M, H, BM) || !make_map(&mb, w, V, H, BN / CL))
    return cudaErrorInvalidValue;
  GemmParams P{};
  P.M = M;
  P.N = V;
  P.K = H;
  P.nm = nm;
  P.nn = (V + BN - 1) / BN;
  P.ntiles = ((P.nm + CL - 1) / CL) * P.nn;  // work units
  P.nkb = (H + BK - 1) / BK;
  P.logits = logits;
  P.ldo = ldo;
  P.stats = (stats && temperature > 0.f) ? stats : nullptr;
  P.kt = temperature > 0.f ? kLog2e / temperature : 0.f;
  P.status = status;
  P.test_stall = test_stall ? 1 : 0;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  auto kern = CL == 2 ? lmhead_gemm<2> : lmhead_gemm<1>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int slots = sms / CL;  // clusters (or CTAs) resident at once
  const int units = P.ntiles < slots ? P.ntiles : slots;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(SPEC_PROF_LMHEAD, st);
  e = cudaLaunchKernelEx(&cfg, kern, ma, mb, P);
  prof_end(SPEC_PROF_LMHEAD, st);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (P.stats && lse) {
    const int rows_per_cta = 8;
    lse_merge<<<(M + rows_per_cta - 1) / rows_per_cta, 32 * rows_per_cta, 0, st>>>(P.stats, M,
                                                                                    P.nn, lse);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace sv
