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
  const float* k_scales;  // FP8 or INT8 cache only
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
  int n_chunk_slots;  // partial slots per (request, query head)
  int chunk_grid;     // decode grid.x: chunk columns, ceil(pages a request can walk /
                      // chunk_pages) (n_chunk_slots without the cascade prefix slots)
  float scale_log2;   // softmax scale * log2(e)
  int tma_rank;       // tensor maps of a 256-byte-row pool: 3 (one box per tile) or 2
  int warp_units;     // tensor-core decode: one warp per request (every request one chunk)
  // Cascade decode (null group_of otherwise): request b belongs to group group_of[b] (-1:
  // none), whose first prefix_pages[g] logical pages are shared by every member and handled
  // by the prefix kernel in chunks of prefix_chunk_pages; their partials take chunk slots
  // 0 .. ceil(prefix_pages[g] / prefix_chunk_pages) - 1 and the request's own pages follow.
  const int32_t* group_of;
  const int32_t* prefix_pages;
  const int32_t* own_start;  // [batch] prefix_pages[group_of[b]] (0 outside groups), or null
  int n_groups;
  int max_prefix_pages;
  int prefix_chunk_pages;
  // 1: the tensor-core decode is a programmatic dependent launch of the cascade prefix kernel:
  // it reads its own pages while the prefix kernel runs and waits for that grid
  // (griddepcontrol.wait) before it reads any prefix partial
  int prefix_dep;
  // 1 (with prefix_dep): a cascade member's own chunks are written as partials (slots slot0 ..)
  // and the combine kernel merges them with the prefix partials; one thread of the decode
  // grid's first CTA waits for the prefix grid before it exits, so the decode grid -- which the
  // combine waits for -- cannot complete before the prefix kernel
  int defer_fold;
  // balanced split (decode_flat.cu): [batch + 1] pages walked per KV head by the requests
  // before b, written by the decode's first CTA for its combine
  int* flat_pre;
};

// Query rows ((member, query head) pairs) per CTA of the cascade prefix kernel, and the CTAs
// of it that run at once on a GB300 (152 SMs x 3 resident CTAs).
constexpr int kCascadeRows = 64;
constexpr int kCascadeWaveCtas = 152 * 3;
// The same for the tcgen05 prefix kernel (M = 128 rows per CTA, one CTA per SM).
constexpr int kCascadeTcRows = 128;
constexpr int kCascadeTcWaveCtas = 152;

// Members of the cascade groups (prefix kernel only).
struct CascadeArgs {
  const int32_t* group_offsets;  // [n_groups + 1]: members of g are group_members[off[g] .. off[g+1])
  const int32_t* group_members;  // request indices
  int max_members;               // rows per group = members * group size; larger groups are cut
  const int32_t* prefix_ids;     // [n_groups][ids_stride] shared page ids, or null: read the
  int ids_stride;                // first member's table row instead
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
// Balanced split of the tensor-core decode (decode_flat.cu): the CTAs of kFlatWarpsPerCta warps
// resident at once for this call (one wave); the decode on `ctas` CTAs with `cap` partial slots
// per query head; its combine, launched with the same `ctas` and `cap`.
constexpr int kFlatWarpsPerCta = 4;
constexpr int kFlatMaxWarps = 1 << 20;  // bounds the warp count (and partial ids) far from int
constexpr int kFlatMaxBatch = 2048;     // per-request page offsets held in shared memory
cudaError_t decode_flat_wave(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                             int* ctas);
cudaError_t launch_decode_flat(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                               int ctas, int cap, const void* tk, const void* tv,
                               cudaStream_t s);
cudaError_t launch_decode_flat_combine(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                                       int ctas, int cap, cudaStream_t s);
cudaError_t launch_kv_append(const AppendArgs& a, int in_dtype, int cache_dtype, cudaStream_t s);
// cudaMemcpyAsync on stream s, traced under `name` when launch tracing is on (capi.cu).
cudaError_t traced_copy(const char* name, void* dst, const void* src, size_t bytes,
                        cudaMemcpyKind kind, cudaStream_t s);
cudaError_t launch_copy_pages(void* k, void* v, const int32_t* src, const int32_t* dst, int n,
                              int64_t page_bytes, int num_pages, int* err, cudaStream_t s);
cudaError_t launch_kv_absmax(const void* x, int dtype, int64_t n_tokens, int h_kv, int head_dim,
                             float code_max, float* scales_out, cudaStream_t s);
// Shared-prefix pass of the cascade decode (bf16 cache and queries, head_dim 128).
cudaError_t launch_cascade_prefix(const DecodeArgs& a, const CascadeArgs& ca, int group,
                                  const void* tk, const void* tv, cudaStream_t s);
// The same pass on tcgen05 (accumulators in tensor memory).
cudaError_t launch_cascade_prefix_tc(const DecodeArgs& a, const CascadeArgs& ca, int group,
                                     const void* tk, const void* tv, cudaStream_t s);
cudaError_t launch_decode_int8(const DecodeArgs& a, int q_dtype, int head_dim, int group,
                               cudaStream_t s);

}  // namespace pkv
