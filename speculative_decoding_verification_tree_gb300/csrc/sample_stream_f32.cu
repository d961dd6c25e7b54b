// Instantiations of the streaming sampled verifier for float32 target logits
// (float32 or bfloat16 draft rows), and its geometry.
#include "sample_stream.cuh"

namespace sv {

cudaError_t launch_stream_f32(StreamParams P, cudaStream_t st) {
  if (P.a.dt_draft == SPEC_BF16) return stream::launch_dt<float, uint16_t>(P, st);
  return stream::launch_dt<float, float>(P, st);
}

bool stream_geometry(int V, int tsz, int dsz, int* C, int* slice, int* nch, int* stages,
                     int64_t rows, int sms, int passA) {
  return stream::geometry(V, tsz, dsz, C, slice, nch, stages, rows, sms, passA);
}

}  // namespace sv
