// Instantiations of the streaming sampled verifier for bfloat16 target
// logits (float32 or bfloat16 draft rows).
#include "sample_stream.cuh"

namespace sv {

cudaError_t launch_stream_bf16(StreamParams P, cudaStream_t st) {
  if (P.a.dt_draft == SPEC_BF16) return stream::launch_dt<uint16_t, uint16_t>(P, st);
  return stream::launch_dt<uint16_t, float>(P, st);
}

}  // namespace sv
