// Decode attention instantiations for an fp32 cache (fp32 queries and output).
#include "paged_decode.cuh"

namespace pkv {
cudaError_t launch_decode_f32(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                              cudaStream_t s) {
  if (q_dtype != PKV_F32) return cudaErrorInvalidValue;
  return launch_decode_d<F32, float>(a, head_dim, group, s);
}
}  // namespace pkv
