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
// Organisation (head dim 128, bf16 inputs, float32 accumulation) on the
// fifth-generation tensor cores.  A CTA takes up to 256 query rows of one
// (sequence, key/value head) -- the rows are (node, head in the group) pairs,
// node-major, so the G query heads that share a key/value head are served by
// one stream of its keys and values -- as two 128-row tiles:
//   warp 0     TMA producer: 64-key blocks of K and V (128-byte swizzle) into
//              a 5-stage shared-memory ring (and a prefetch into L2 of the
//              block that will next fill the stage it waits for);
//   warps 1-2  tile t's S issuer (warp 1 also allocates TMEM): S_t = Q_t K^T
//              of each key block (tcgen05.mma M 128, N 64, K 128, Q_t read
//              from TMEM, K from shared memory) once the block's keys have
//              landed and the softmax has read S_t of the block before;
//   warps 3-4  tile t's P V issuer: O_t += P_t V of each block (M 128,
//              N 128, K 64; V is the MN-major operand, read as stored) once
//              the softmax has written P_t -- four issuing threads, so that
//              neither tile and neither chain of issues waits on another;
//   warps 5-12 softmax, one thread per query row (warp w reads TMEM lanes of
//              quadrant w % 4): they write their row of Q into TMEM once, then
//              per block read S with tcgen05.ld, apply the scale and the tree
//              mask, run the online base-2 softmax against a reference maximum
//              that moves only when a row's maximum grows by more than 2^8
//              (then O_t is rescaled in TMEM), and write P as bf16 into
//              128-byte-swizzled shared memory for the next MMA (two P
//              buffers per tile, so that block j + 1's P is written while
//              block j's P V runs); at the end O_t / l is rounded to bf16.
// TMEM (512 columns): Q_t at columns 64 t (two bf16 per column), S_t at
// 128 + 64 t, O_t at 256 + 128 t.  With Q in TMEM the tensor cores read only
// K (2 KB per MMA instead of 6) from shared memory for S, and shared memory
// holds the 5-stage ring and two P buffers per tile (224 KB).  Every
// mbarrier wait is bounded (SPEC_STATUS_TIMEOUT is not reported by this
// entry point, which has no status word; a CTA that gives up stops waiting
// and still frees its TMEM after waiting, bounded, for its own MMAs and
// copies).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr int kAD = 128;   // head dim
constexpr int kKB = 64;    // keys per block
constexpr int kMT = 128;   // query rows per tile
constexpr int kTiles = 2;  // tiles per CTA
constexpr int kAStages = 5;
constexpr int kKVHalf = kKB * 64 * 2;    // 8 KB: 64 keys x 64 dims
constexpr int kKVTile = 2 * kKVHalf;     // 16 KB
constexpr int kAStage = 2 * kKVTile;     // K then V: 32 KB
constexpr int kPTile = kMT * kKB * 2;    // 16 KB: 128 rows x 64 keys
constexpr int kOffKV = 0;
constexpr int kOffP = kOffKV + kAStages * kAStage;       // 160 KB
constexpr int kOffBar = kOffP + kTiles * 2 * kPTile;     // 224 KB: two P buffers per tile
constexpr int kAThreads = 416;
constexpr int kPrefetch = 0;  // key blocks prefetched into L2 ahead of the ring
constexpr int kSoftThreads = 256;
constexpr uint32_t kATmemCols = 512;
constexpr int kOrderMax = 256;  // sequences ordered longest first up to this batch

struct __align__(8) AttnSmem {
  uint64_t kvfull[kAStages], kvempty[kAStages];
  uint64_t sfull[kTiles], sfree[kTiles], pfull[kTiles][2], pdone[kTiles][2];
  uint64_t qready, drain[kTiles][2];
  uint32_t tmem_base;
  uint32_t dead;
  int seq;
};
constexpr size_t kASmemBytes = (size_t)kOffBar + sizeof(AttnSmem) + 1024;

// S = Q K^T: M 128, N 64, bf16 K-major A (in TMEM) and B, float32 D.
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kKB >> 3) << 17) |
                             ((uint32_t)(kMT >> 4) << 24);
// O += P V: M 128, N 128, A K-major, B MN-major (bit 16).
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              ((uint32_t)(kAD >> 3) << 17) | ((uint32_t)(kMT >> 4) << 24);

__device__ __forceinline__ void await(AttnSmem& sm, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  if (*(volatile uint32_t*)&sm.dead) return;
  if (!mbar_wait_bounded(bar, parity)) *(volatile uint32_t*)&sm.dead = 1;
}

// K-major tile with 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups
// 1024 B apart (start 1024-byte aligned; K steps add 32 B within a row).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// MN-major tile with 128-byte swizzle (V as stored: a key per 128-byte row of
// 64 head dims): 64-dim column blocks kKVHalf apart (leading offset), 8-key
// groups 1024 B apart (stride offset); K steps of 16 keys add 2048 B.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kKVHalf >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                      uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma2d_prefetch(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// the same with A read from TMEM (column address a; two bf16 per column,
// the lower K index in the low half)
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// generic-proxy shared-memory writes made visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define SV_R32(r)                                                                          \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),         \
      "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),      \
      "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),      \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),      \
      "=r"(r[31])
#define SV_W32(r)                                                                            \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),     \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),   \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),   \
      "r"(r[29]), "r"(r[30]), "r"(r[31])
#define SV_REGS32                                                     \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
  "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}"

__device__ __forceinline__ void tld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " SV_REGS32 ", [%32];"
               : SV_R32(r)
               : "r"(taddr));
}
__device__ __forceinline__ void tst32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
               "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
               "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
               SV_W32(r)
               : "memory");
}
__device__ __forceinline__ void tld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tst_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// two floats -> bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled block
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kAThreads, 1)
    tree_attn_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const uint16_t* __restrict__ q, const int32_t* __restrict__ prefix_len,
                 const uint64_t* __restrict__ mask_bits, int N, int Hq, int Hkv, int S,
                 float scale_log2, uint16_t* __restrict__ out) {
  extern __shared__ __align__(1024) unsigned char araw[];
  const uint32_t raw = smem_u32(araw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* bp = araw + (base - raw);
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(bp + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / Hkv, R = N * G;
  int b = blockIdx.z, kvh = blockIdx.y, tile = blockIdx.x;
  if (gridDim.z <= (unsigned)kOrderMax) {
    // longest sequences first: the CTAs launched first (lowest linear index)
    // take the sequences with the most keys, so the last CTAs to start are
    // the shortest ones and the tail of the grid is short
    const int nb = (int)gridDim.z, gx = (int)gridDim.x;
    const int lin = blockIdx.x + gx * (blockIdx.y + Hkv * blockIdx.z);
    const int want = lin / (gx * Hkv), rem = lin % (gx * Hkv);
    int* len_s = reinterpret_cast<int*>(bp + kOffP);  // P tiles are written later
    for (int i = threadIdx.x; i < nb; i += kAThreads) {
      const int p = prefix_len[i];
      len_s[i] = p < 0 ? 0 : (p > S - N ? S - N : p);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb; i += kAThreads) {
      const int li = len_s[i];
      int rank = 0;
      for (int j = 0; j < nb; ++j) {
        const int lj = len_s[j];
        rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
      }
      if (rank == want) sm.seq = i;
    }
    __syncthreads();
    b = sm.seq;
    kvh = rem / gx;
    tile = rem % gx;
  }
  const int row0 = tile * (kTiles * kMT);
  const int ntile = min(kTiles, (R - row0 + kMT - 1) / kMT);
  int P = prefix_len[b];
  P = P < 0 ? 0 : (P > S - N ? S - N : P);
  const int L = P + N;
  const int nblk = (L + kKB - 1) / kKB;
  const int kvrow0 = (b * Hkv + kvh) * S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&sm.kvfull[s], 1);
      mbar_init(&sm.kvempty[s], ntile);  // released by every tile's issuer
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&sm.sfull[t], 1);
      mbar_init(&sm.sfree[t], kMT);
      mbar_init(&sm.pfull[t][0], kMT);
      mbar_init(&sm.pfull[t][1], kMT);
      mbar_init(&sm.pdone[t][0], 1);
      mbar_init(&sm.pdone[t][1], 1);
    }
    mbar_init(&sm.qready, kSoftThreads);
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&sm.drain[t][0], 1);
      mbar_init(&sm.drain[t][1], 1);
    }
    sm.dead = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem_base)),
                 "r"(kATmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto prefetch = [&](int j) {
        const int y = kvrow0 + j * kKB;
        tma2d_prefetch(&map_k, 0, y);
        tma2d_prefetch(&map_k, 64, y);
        tma2d_prefetch(&map_v, 0, y);
        tma2d_prefetch(&map_v, 64, y);
      };
      for (int j = kAStages; j < kAStages + kPrefetch && j < nblk; ++j) prefetch(j);
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kAStages;
        if (j + kAStages + kPrefetch < nblk) prefetch(j + kAStages + kPrefetch);
        await(sm, &sm.kvempty[s], ((uint32_t)(j / kAStages) & 1u) ^ 1u);
        mbar_expect_tx(&sm.kvfull[s], (uint32_t)kAStage);
        const uint32_t st = base + kOffKV + (uint32_t)(s * kAStage);
        const int y = kvrow0 + j * kKB;
        tma2d(st, &map_k, 0, y, &sm.kvfull[s]);
        tma2d(st + kKVHalf, &map_k, 64, y, &sm.kvfull[s]);
        tma2d(st + kKVTile, &map_v, 0, y, &sm.kvfull[s]);
        tma2d(st + kKVTile + kKVHalf, &map_v, 64, y, &sm.kvfull[s]);
      }
      // this CTA's last copy into each stage has landed before it exits
      for (int s = 0; s < kAStages && s < nblk; ++s) {
        const int fills = (nblk - s + kAStages - 1) / kAStages;
        mbar_wait_bounded(&sm.kvfull[s], (uint32_t)(fills - 1) & 1u);
      }
    }
  } else if (warp <= 2) {
    // ------------------------------------------------ tile t's S issuer
    // Warp 1 + t issues S_t = Q_t K^T of each block as soon as its keys have
    // landed and the softmax has read S_t of the block before.
    const int t = warp - 1;
    if (lane == 0 && t < ntile) {
      await(sm, &sm.qready, 0);
      fence_after();
      const uint32_t tq = tmem + (uint32_t)(64 * t);
      const uint32_t ds = tmem + 128u + (uint32_t)(64 * t);
      // descriptors are formed once: shared-memory addresses here stay below
      // 256 KB, so a byte offset (a multiple of 16) adds offset / 16 to the
      // 14-bit address field
      const uint64_t dk0 = desc_kmajor(base + kOffKV);
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kAStages;
        await(sm, &sm.kvfull[s], (uint32_t)(j / kAStages) & 1u);
        // S_t was last read by the softmax at block j - 1
        if (j >= 1) await(sm, &sm.sfree[t], (uint32_t)((j - 1) & 1));
        fence_after();
        const uint64_t dk = dk0 + (uint64_t)((s * kAStage) >> 4);
        // K step k: head dims 16k .. 16k + 15 = Q_t's TMEM columns 8k .. 8k + 7
#pragma unroll
        for (int k = 0; k < kAD / 16; ++k) {
          const uint32_t koff = (uint32_t)((k >> 2) * kKVHalf + (k & 3) * 32);
          mma_f16_ts(ds, tq + (uint32_t)(8 * k), dk + (koff >> 4), kIdescS, k > 0 ? 1u : 0u);
        }
        mma_commit(&sm.sfull[t]);
      }
      mma_commit(&sm.drain[t][0]);
      mbar_wait_bounded(&sm.drain[t][0], 0);
    }
  } else if (warp <= 4) {
    // --------------------------------------------- tile t's P V issuer
    // Warp 3 + t issues O_t += P_t V of each block as soon as the softmax
    // has written P_t (a separate thread from the S issuer, so that neither
    // chain of issues waits behind the other).
    const int t = warp - 3;
    if (lane == 0 && t < ntile) {
      // descriptors formed once (see the S issuer)
      const uint64_t dv0 = desc_mnmajor(base + kOffKV + kKVTile);
      const uint64_t dp0 = desc_kmajor(base + kOffP + (uint32_t)(2 * t * kPTile));
      const uint32_t to = tmem + 256u + (uint32_t)(128 * t);
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kAStages;
        const int tail = L - j * kKB;  // keys of this block that exist
        if (tail < kKB) {
          // cache rows past the sequence's keys hold anything (NaN included);
          // their P is 0, but 0 * NaN is not, so their V rows become zeros
          // (each tile's issuer writes the same zeros before its own MMAs),
          // after the block's copy has landed
          await(sm, &sm.kvfull[s], (uint32_t)(j / kAStages) & 1u);
          unsigned char* vz = bp + kOffKV + s * kAStage + kKVTile;
          for (int rr = tail; rr < kKB; ++rr)
            for (int hb = 0; hb < 2; ++hb) {
              uint4* z = reinterpret_cast<uint4*>(vz + hb * kKVHalf + rr * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          fence_async_smem();
        }
        await(sm, &sm.pfull[t][j & 1], (uint32_t)((j >> 1) & 1));
        fence_after();
        const uint64_t dp = dp0 + (uint64_t)(((j & 1) * kPTile) >> 4);
        const uint64_t dv = dv0 + (uint64_t)((s * kAStage) >> 4);
#pragma unroll
        for (int k = 0; k < kKB / 16; ++k)
          mma_f16(to, dp + (uint64_t)(k * 2), dv + (uint64_t)(k * 128), kIdescPV,
                  (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(&sm.pdone[t][j & 1]);
        // this tile is done with the block's K and V (its S MMAs completed
        // before the softmax wrote P)
        mma_commit(&sm.kvempty[s]);
      }
      mma_commit(&sm.drain[t][1]);
      mbar_wait_bounded(&sm.drain[t][1], 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int t = (warp - 5) >> 2;   // tile
    const int qd = warp & 3;         // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;    // row within the tile
    const int gr = row0 + t * kMT + r;
    const bool valid = t < ntile && gr < R;
    const int node = valid ? gr / G : 0;
    const int hq = kvh * G + (valid ? gr % G : 0);
    const uint64_t mb = valid ? (mask_bits[(int64_t)b * N + node] &
                                 (N >= 64 ? ~0ull : ((1ull << N) - 1ull)))
                              : 0ull;
    const int64_t qoff = (((int64_t)b * N + node) * Hq + hq) * kAD;
    const uint32_t lanes = (uint32_t)(qd * 32) << 16;
    {  // this row of Q into Q_t's TMEM lane (zeros for padding rows)
      const uint4* src = reinterpret_cast<const uint4*>(q + qoff);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = valid ? src[8 * h + c] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tst32(tmem + lanes + (uint32_t)(64 * t + 32 * h), w);
      }
      tst_wait();
      fence_before();
      mbar_arrive(&sm.qready);
    }
    if (t < ntile) {
      const uint32_t tS = tmem + lanes + 128u + (uint32_t)(64 * t);
      const uint32_t tO = tmem + lanes + 256u + (uint32_t)(128 * t);
      unsigned char* pt0 = bp + kOffP + 2 * t * kPTile;
      float mref = neg_inf(), l = 0.f;
      for (int j = 0; j < nblk; ++j) {
        await(sm, &sm.sfull[t], (uint32_t)(j & 1));
        fence_after();
        uint32_t ra[32], rb[32];
        tld32(tS, ra);
        tld32(tS + 32u, rb);
        tld_wait();
        fence_before();
        mbar_arrive(&sm.sfree[t]);  // the S issuer may write S_t of the next block
        // raw scores q.k (the scale is applied inside the exponent below;
        // it is positive, so the maximum is taken on the raw scores)
        float s[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(ra[i]);
          s[32 + i] = __uint_as_float(rb[i]);
        }
        const int key0 = j * kKB;
        if (!valid || key0 + kKB > P) {
          // visibility of the block's 64 keys as one word: the prefix (keys
          // < P) and the drafted keys P + i whose bit i is set in the node's
          // mask row (its ancestors and itself; bits only below N)
          const int npre = min(max(P - key0, 0), 64);
          const uint64_t pre = npre >= 64 ? ~0ull : ((1ull << npre) - 1ull);
          const int off = key0 - P;
          const uint64_t dr = off >= 0 ? (off < 64 ? (mb >> off) : 0ull)
                                       : (off > -64 ? (mb << (-off)) : 0ull);
          const uint64_t vis = valid ? (pre | dr) : 0ull;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (!((vis >> i) & 1ull)) s[i] = neg_inf();
        }
        // four independent chains of three-input maxima, then their combination
        float bm4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) bm4[c] = fmax3f(s[c], s[c + 4], s[c + 8]);
#pragma unroll
        for (int i = 12; i < 60; i += 8)
#pragma unroll
          for (int c = 0; c < 4; ++c) bm4[c] = fmax3f(bm4[c], s[i + c], s[i + 4 + c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) bm4[c] = fmaxf(bm4[c], s[60 + c]);
        const float bm = fmaxf(fmax3f(bm4[0], bm4[1], bm4[2]), bm4[3]) * scale_log2;
        // the reference maximum moves only when the row's maximum grows by
        // more than 2^8 (also at the first visible key): P stays below 2^8
        const bool move = bm > mref + 8.f;
        const float mnew = move ? bm : mref;
        const float corr = (move && mref != neg_inf()) ? ex2(mref - mnew) : 1.f;
        mref = mnew;
        const float nmu = mref == neg_inf() ? 0.f : -mref;
        // exponents and the row sum on packed pairs
        uint32_t pk[32];
        const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(nmu, nmu);
        float2 ls4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 e = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sc2, nm2);
          const float p0 = ex2(e.x), p1 = ex2(e.y);
          ls4[i & 3] = fadd2(ls4[i & 3], make_float2(p0, p1));
          pk[i] = pack_bf16(p0, p1);
        }
        const float2 lsa = fadd2(fadd2(ls4[0], ls4[1]), fadd2(ls4[2], ls4[3]));
        const float ls = lsa.x + lsa.y;
        l = l * corr + ls;
        // P buffer j & 1 was read by the P V of block j - 2, which must be
        // done before it is rewritten; a rescale of O_t needs the P V of
        // block j - 1 done too (a commit covers every earlier MMA of its
        // issuer, so that wait covers both)
        const bool resc = j > 0 && __any_sync(0xffffffffu, corr != 1.f);
        if (resc)
          await(sm, &sm.pdone[t][(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1));
        else if (j >= 2)
          await(sm, &sm.pdone[t][j & 1], (uint32_t)(((j - 2) >> 1) & 1));
        fence_after();
        if (resc) {
#pragma unroll 1
          for (int c = 0; c < kAD / 32; ++c) {
            uint32_t o[32];
            tld32(tO + (uint32_t)(32 * c), o);
            tld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tst32(tO + (uint32_t)(32 * c), o);
          }
          tst_wait();
        }
        unsigned char* pt = pt0 + (j & 1) * kPTile;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(pt + swz(r, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_async_smem();
        fence_before();
        mbar_arrive(&sm.pfull[t][j & 1]);
      }
      // O_t / l after the last P V
      if (nblk > 0)
        await(sm, &sm.pdone[t][(nblk - 1) & 1], (uint32_t)(((nblk - 1) >> 1) & 1));
      fence_after();
      const float inv = 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(out + qoff);
#pragma unroll 1
      for (int c = 0; c < kAD / 32; ++c) {
        uint32_t o[32];
        tld32(tO + (uint32_t)(32 * c), o);
        tld_wait();
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int i = 8 * v;
            dst[4 * c + v] = make_uint4(
                pack_bf16(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv),
                pack_bf16(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv),
                pack_bf16(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv),
                pack_bf16(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv));
          }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kATmemCols)
                 : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A cache [rows, 128] bf16 as 64-dim x 64-key boxes, 128-byte swizzle.
bool cache_map(CUtensorMap* map, const void* base, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kAD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kAD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kKB};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  // rows of q / out are read and written as 16-byte words
  if (((uintptr_t)q | (uintptr_t)out) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)B * Hkv * S;
  if (rows > ((int64_t)1 << 31) - kKB) return SPEC_ERR_SHAPE;
  CUtensorMap mk, mv;
  if (!cache_map(&mk, k_cache, rows) || !cache_map(&mv, v_cache, rows)) return SPEC_ERR_CUDA;
  const int R = N * (Hq / Hkv);
  const dim3 grid((unsigned)((R + kTiles * kMT - 1) / (kTiles * kMT)), (unsigned)Hkv, (unsigned)B);
  if (cudaFuncSetAttribute(tree_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kASmemBytes) != cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  prof_begin(SPEC_PROF_ATTN, st);
  tree_attn_tc<<<grid, kAThreads, kASmemBytes, st>>>(
      mk, mv, (const uint16_t*)q, prefix_len, mask_bits, N, Hq, Hkv, S, scale * kLog2e,
      (uint16_t*)out);
  prof_end(SPEC_PROF_ATTN, st);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
