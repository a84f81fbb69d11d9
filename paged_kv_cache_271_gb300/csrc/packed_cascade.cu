// The cascade decode step from host memory: the step's inputs packed in one pinned host block
// (as for pkv_paged_decode_step_packed) plus room for the batch's groups, which this call finds
// on the host from the packed page tables ("KV cache and PagedAttention", section 6: requests
// with a common prompt share its pages). One host-to-device copy of the block, the cascade
// step on the device copies, one device-to-host copy of the output. Built from the library's
// C entry points (grouping, workspace size, cascade step) and its traced copy.
#include <cuda_runtime.h>

#include <cstring>

#include "pkv.h"
#include "pkv_host.h"
#include "pkv_internal.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

int pkv_packed_cascade_layout(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_pages_per_seq, int32_t dtype_q,
                              int32_t dtype_new, size_t* offsets, size_t* total_bytes) {
  if (!offsets || !total_bytes)
    return pkv::set_error(PKV_EINVAL, "pkv_packed_cascade_layout: bad argument");
  size_t base = 0;
  int st = pkv_packed_step_layout(batch, num_q_heads, num_kv_heads, head_dim, max_pages_per_seq,
                                  dtype_q, dtype_new, offsets, &base);
  if (st != PKV_OK) return st;
  // group_of [B], prefix_pages [B], group_offsets [B + 1], group_members [B], own_start [B],
  // the groups' shared page ids [B / 2][max_pages] (last: a step copies only what it uses)
  const size_t words[6] = {(size_t)batch, (size_t)batch, (size_t)batch + 1, (size_t)batch,
                           (size_t)batch, (size_t)(batch / 2) * max_pages_per_seq};
  size_t off = base;
  for (int i = 0; i < 6; ++i) {
    offsets[5 + i] = off;
    off += align256(words[i] * 4);
  }
  *total_bytes = off;
  return PKV_OK;
}

int pkv_cascade_decode_step_packed(void* host_in, void* dev_in, int32_t batch,
                                   int32_t num_q_heads, int32_t dtype_q, int32_t dtype_new,
                                   void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                   int32_t max_pages_per_seq, float scale, void* out_dev,
                                   void* out_host, void* workspace, size_t workspace_bytes,
                                   size_t* workspace_needed, int32_t* n_groups_out,
                                   void* stream) {
  const char* who = "pkv_cascade_decode_step_packed";
  if (!desc) return pkv::set_error(PKV_EINVAL, "%s: desc is NULL", who);
  size_t off[11], total = 0;
  int st = pkv_packed_cascade_layout(batch, num_q_heads, desc->num_kv_heads, desc->head_dim,
                                     max_pages_per_seq, dtype_q, dtype_new, off, &total);
  if (st != PKV_OK) return st;
  if (batch == 0) return PKV_OK;  // (an empty batch may pass null buffers)
  if (!host_in || !dev_in || !out_dev || !out_host)
    return pkv::set_error(PKV_EINVAL, "%s: null pointer", who);
  char* h = static_cast<char*>(host_in);
  char* d = static_cast<char*>(dev_in);
  auto hp = [&](int i) { return reinterpret_cast<int32_t*>(h + off[i]); };
  auto dp = [&](int i) { return reinterpret_cast<const int32_t*>(d + off[i]); };
  // this step's groups, from the host tables, into the block before it is copied
  int32_t n_groups = 0, max_members = 0, max_prefix = 0, max_own = 0;
  st = pkv_cascade_groups(hp(3), hp(4), batch, max_pages_per_seq, 2, 1, hp(5), hp(6), hp(7),
                          hp(8), &n_groups, &max_members, &max_prefix, &max_own, hp(9));
  if (st != PKV_OK) return st;
  if (n_groups_out) *n_groups_out = n_groups;
  pkv_cascade_desc g;
  std::memset(&g, 0, sizeof(g));
  g.n_groups = n_groups;
  if (n_groups > 0) {
    g.group_of = dp(5);
    g.prefix_pages = dp(6);
    g.group_offsets = dp(7);
    g.group_members = dp(8);
    g.own_start = dp(9);
    g.max_members = max_members;
    g.max_prefix_pages = max_prefix;
    g.max_own_pages = max_own;
    st = pkv_cascade_prefix_page_ids(hp(3), batch, max_pages_per_seq, hp(6), hp(7), hp(8),
                                     n_groups, max_prefix, hp(10));
    if (st != PKV_OK) return st;
    g.prefix_page_ids = dp(10);
  }
  const size_t need = pkv_cascade_workspace_size(batch, num_q_heads, desc->num_kv_heads,
                                                 desc->head_dim, max_pages_per_seq, &g);
  if (workspace_needed) *workspace_needed = need;
  if (need > 0 && (!workspace || workspace_bytes < need))
    return pkv::set_error(PKV_EINVAL, "%s: workspace of %zu bytes needed, %zu given", who, need,
                          workspace_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the block up to the end of the page ids this step's groups use
  const size_t used = off[10] + (size_t)n_groups * max_prefix * sizeof(int32_t);
  cudaError_t e = pkv::traced_copy("h2d_copy", dev_in, host_in, used, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess)
    return pkv::set_error(PKV_ECUDA, "%s: input copy: %s", who, cudaGetErrorString(e));
  st = pkv_cascade_decode_step(d + off[0], dtype_q, batch, num_q_heads, d + off[1], d + off[2],
                               dtype_new, k_cache, v_cache, desc, dp(3), max_pages_per_seq,
                               dp(4), scale, &g, out_dev, workspace, workspace_bytes, stream);
  if (st != PKV_OK) return st;
  const size_t out_bytes =
      (size_t)batch * num_q_heads * desc->head_dim * (dtype_q == PKV_F32 ? 4 : 2);
  e = pkv::traced_copy("d2h_copy", out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess)
    return pkv::set_error(PKV_ECUDA, "%s: output copy: %s", who, cudaGetErrorString(e));
  return PKV_OK;
}

}  // extern "C"
