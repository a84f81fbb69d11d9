// Tensor-core decode attention instantiations (bf16 cache with bf16 queries; FP8 or INT8 cache
// with bf16 or fp32 queries), head_dim 128, groups 1..16.
#include "paged_decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_mma(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                              const void* tk, const void* tv, cudaStream_t s) {
  const CUtensorMap& k = *static_cast<const CUtensorMap*>(tk);
  const CUtensorMap& v = *static_cast<const CUtensorMap*>(tv);
  if (kv_dtype == PKV_BF16 && q_dtype == PKV_BF16)
    return launch_decode_mma_g<BF16, __nv_bfloat16>(a, group, k, v, s);
  if (kv_dtype == PKV_FP8_E4M3 && q_dtype == PKV_BF16)
    return launch_decode_mma_g<FP8, __nv_bfloat16>(a, group, k, v, s);
  if (kv_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F32)
    return launch_decode_mma_g<FP8, float>(a, group, k, v, s);
  if (kv_dtype == PKV_INT8 && q_dtype == PKV_BF16)
    return launch_decode_mma_g<INT8, __nv_bfloat16>(a, group, k, v, s);
  if (kv_dtype == PKV_INT8 && q_dtype == PKV_F32)
    return launch_decode_mma_g<INT8, float>(a, group, k, v, s);
  return cudaErrorInvalidValue;
}
}  // namespace pkv
