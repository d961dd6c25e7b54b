// Instantiations of the pipelined sampled-verification kernel for float32
// target logits, and the walk that follows it.
#include "sample_pipe.cuh"

namespace sv {

cudaError_t launch_pipe_f32(const PipeParams& P, int C, int ept, int qk, int dt_draft,
                            cudaStream_t st) {
  if (dt_draft == SPEC_BF16) return pipe::launch_pipe_dt<float, uint16_t>(P, C, ept, qk, st);
  return pipe::launch_pipe_dt<float, float>(P, C, ept, qk, st);
}

cudaError_t launch_pipe_walk(const VerifyShape& s, const VerifyArgs& a, int C, cudaStream_t st) {
  const int64_t rows = s.rows();
  pipe::pipe_walk<<<(unsigned)((rows + 127) / 128), 128, 0, st>>>(s, a, C);
  return cudaGetLastError();
}

bool pipe_geometry(int V, int tsz, int dsz, int* C, int* ept, int* stages, int* slice) {
  return pipe::geometry(V, tsz, dsz, C, ept, stages, slice);
}

}  // namespace sv
