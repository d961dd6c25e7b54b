// Tree attention mask (EAGLE-2 notes §4.2, verification input and its mask):
// a drafted token sees only itself and its ancestors; for a chain this is the
// lower-triangular causal mask.  Parents precede children, so row i of the
// mask is row parent(i) plus the diagonal bit, and the rows can be built in
// node order with all threads of the CTA sweeping the columns.
//
// Also: the device side of spec_philox_uniforms.
#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

__global__ void __launch_bounds__(256) tree_mask_kernel(const int32_t* __restrict__ parent, int N,
                                                        uint8_t* __restrict__ mask,
                                                        uint64_t* __restrict__ bits) {
  const int b = blockIdx.x;
  const int32_t* par = parent + (int64_t)b * N;
  if (mask) {
    uint8_t* m = mask + (int64_t)b * N * N;
    for (int i = 0; i < N; ++i) {
      const int p = par[i];
      const bool ok = (p >= 0 && p < i);
      uint8_t* row = m + (int64_t)i * N;
      const uint8_t* prow = m + (int64_t)(ok ? p : 0) * N;
      for (int j = threadIdx.x; j < N; j += blockDim.x)
        row[j] = (j == i) ? 1 : (ok && j < i ? prow[j] : 0);
      __syncthreads();  // row i is read when its children are built
    }
  }
  if (bits && threadIdx.x == 0) {
    uint64_t* o = bits + (int64_t)b * N;
    for (int i = 0; i < N; ++i) {
      const int p = par[i];
      const uint64_t up = (p >= 0 && p < i) ? o[p] : 0ull;
      o[i] = up | (1ull << i);
    }
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
