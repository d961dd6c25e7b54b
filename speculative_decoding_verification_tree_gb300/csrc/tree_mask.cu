// Tree attention mask (EAGLE-2 notes §4.2, verification input and its mask):
// a drafted token sees only itself and its ancestors; for a chain this is the
// lower-triangular causal mask.  One CTA per sequence: the parent array goes
// to shared memory, the N x N block is zeroed, then one thread per row walks
// the row's ancestor chain (parents precede children; a link that does not
// point to an earlier node ends the chain) and sets those bytes.
//
// Also: the device side of spec_philox_uniforms.
#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

__global__ void __launch_bounds__(256) tree_mask_kernel(const int32_t* __restrict__ parent, int N,
                                                        uint8_t* __restrict__ mask,
                                                        uint64_t* __restrict__ bits) {
  __shared__ int par[SPEC_MAX_TREE_NODES];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < N; i += blockDim.x) par[i] = parent[(int64_t)b * N + i];
  uint8_t* m = mask ? mask + (int64_t)b * N * N : nullptr;
  if (m)
    for (int k = threadIdx.x; k < N * N; k += blockDim.x) m[k] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    uint64_t w = 0;
    if (m) m[(int64_t)i * N + i] = 1;
    if (i < 64) w = 1ull << i;
    int cur = i, a = par[i];
    while (a >= 0 && a < cur) {
      if (m) m[(int64_t)i * N + a] = 1;
      if (a < 64) w |= 1ull << a;
      cur = a;
      a = par[a];
    }
    if (bits) bits[(int64_t)b * N + i] = w;
  }
}

__global__ void philox_kernel(uint64_t seed, uint32_t offset, const int32_t* b, const int32_t* i,
                              const int32_t* slot, int n, float* out) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k < n) out[k] = philox_uniform(seed, offset, (uint32_t)b[k], (uint32_t)i[k], (uint32_t)slot[k]);
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parent, int B, int N, uint8_t* mask, uint64_t* bits,
                             cudaStream_t st) {
  if (B == 0 || N == 0) return cudaSuccess;
  tree_mask_kernel<<<B, 256, 0, st>>>(parent, N, mask, bits);
  return cudaGetLastError();
}

cudaError_t launch_philox(uint64_t seed, uint32_t offset, const int32_t* b, const int32_t* i,
                          const int32_t* slot, int n, float* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  philox_kernel<<<(n + 255) / 256, 256, 0, st>>>(seed, offset, b, i, slot, n, out);
  return cudaGetLastError();
}

}  // namespace sv
