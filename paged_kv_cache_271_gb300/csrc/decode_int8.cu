// Decode attention instantiations (CUDA cores) for an INT8 cache (fp32 or bf16 queries).
#include "paged_decode.cuh"

namespace pkv {
cudaError_t launch_decode_int8(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                               cudaStream_t s) {
  if (q_dtype == PKV_BF16) return launch_decode_d<INT8, __nv_bfloat16>(a, head_dim, group, s);
  if (q_dtype == PKV_F32) return launch_decode_d<INT8, float>(a, head_dim, group, s);
  return cudaErrorInvalidValue;
}
}  // namespace pkv
