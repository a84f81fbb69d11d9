// Decode attention instantiations for a bf16 cache (bf16 queries and output).
#include "paged_decode.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                               cudaStream_t s) {
  if (q_dtype != PKV_BF16) return cudaErrorInvalidValue;
  return launch_decode_d<BF16, __nv_bfloat16>(a, head_dim, group, s);
}
}  // namespace pkv
