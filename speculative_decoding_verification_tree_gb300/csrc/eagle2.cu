// EAGLE-2 expand / rerank (EAGLE-2 notes §4.1-4.2).
#include "common.cuh"
#include "kernels.h"

namespace sv {

cudaError_t launch_eagle2(const void*, int, int, int, int, int, int, int, float, int32_t*,
                          int32_t*, int32_t*, float*, uint8_t*, Eagle2Cand*, uint32_t*,
                          cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace sv
