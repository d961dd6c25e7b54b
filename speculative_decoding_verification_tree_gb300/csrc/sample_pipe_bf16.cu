// Instantiations of the pipelined sampled-verification kernel for bfloat16
// target logits (float32 or bfloat16 draft rows).
#include "sample_pipe.cuh"

namespace sv {

cudaError_t launch_pipe_bf16(const PipeParams& P, int C, int ept, int qk, int dt_draft,
                             cudaStream_t st) {
  if (dt_draft == SPEC_BF16) return pipe::launch_pipe_dt<uint16_t, uint16_t>(P, C, ept, qk, st);
  return pipe::launch_pipe_dt<uint16_t, float>(P, C, ept, qk, st);
}

}  // namespace sv
