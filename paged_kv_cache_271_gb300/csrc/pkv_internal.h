// Internal interface between the C-ABI layer (capi.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

struct DecodeArgs {
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scales;  // FP8 cache only
  const float* v_scales;
  float* ws_acc;  // [batch][h_q][n_chunk_slots][D] partial weighted values (split only)
  float* ws_ml;   // [batch][h_q][n_chunk_slots][2] partial (max, sum), log2 domain
  int* counters;  // [batch][h_kv] finished-chunk counts (merge in place); zero between calls
  int* err;       // device error word
  const void* k_new;  // decode step only: this step's K/V rows [batch][h_kv][D], else null
  const void* v_new;
  int new_dtype;      // pkv_dtype of k_new / v_new
  int merge_in_place; // 1: the last CTA of each (request, kv head) merges the chunks
  int window;         // > 0: attend only the last `window` positions (plus `sink` first ones)
  int sink;
  int batch;
  int h_q;
  int h_kv;
  int num_pages;
  int max_pages;      // block-table width
  int chunk_pages;    // pages per chunk (one CTA)
  int n_chunk_slots;  // grid.x = ceil(max_pages / chunk_pages)
  float scale_log2;   // softmax scale * log2(e)
};

struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int64_t* slots;
  void* k_cache;
  void* v_cache;
  const float* k_scales;
  const float* v_scales;
  int* err;
  int num_tokens;
  int h_kv;
  int head_dim;
  int64_t num_slots;  // num_pages * page_size
};

// Each returns the launch status. dtype codes are pkv_dtype values.
cudaError_t launch_decode_f32(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                              cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                               cudaStream_t s);
cudaError_t launch_decode_fp8(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                              cudaStream_t s);
// Tensor-core decode (bf16 or FP8 cache, head_dim 128); tk/tv are CUtensorMap objects
// describing the K and V pools as 2-D [rows][head_dim] tensors (see capi.cu).
cudaError_t launch_decode_mma(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                              const void* tk, const void* tv, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeArgs& a, int q_dtype, int head_dim,
                                  cudaStream_t s);
cudaError_t launch_kv_append(const AppendArgs& a, int in_dtype, int cache_dtype, cudaStream_t s);
cudaError_t launch_copy_pages(void* k, void* v, const int32_t* src, const int32_t* dst, int n,
                              int64_t page_bytes, int num_pages, int* err, cudaStream_t s);
cudaError_t launch_kv_absmax(const void* x, int dtype, int64_t n_tokens, int h_kv, int head_dim,
                             float code_max, float* scales_out, cudaStream_t s);
cudaError_t launch_decode_int8(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                               cudaStream_t s);

}  // namespace pkv
