// Decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attention asks its caller for a workspace whenever a sequence is long enough
// to be split into chunks. Some callers have no way to provide one: a plugin living inside a
// host application that owns every byte of device memory and offers it no allocation hook, a
// serving loop that reserved all free HBM for the KV pools at start-up (so any later cudaMalloc
// fails), or a latency-critical path that must not call cudaMalloc because it can synchronise
// the whole device. This entry point serves them: it computes the same attention with the same
// kernels, but keeps the split partials in a fixed scratch array that is part of the library
// image instead of in caller memory.
//
// The scratch is kScratchBytes (16 MiB). It lives in device memory on every GPU where the
// library's device code has been loaded and stays there until the process exits. Its device
// address is looked up once per device, on the first call made with that device current; make
// that first call before starting any stream capture on that device. The address belongs to
// the device's context: after a cudaDeviceReset the next call finds a new context and looks
// the address up again. All calls on a device share
// the one array and it keeps whatever the last call left in it. Each call zeroes the small
// region of per-group chunk counters that must start at zero; the partial results are written
// before they are read. Two calls whose kernels can overlap on the GPU (different streams without ordering
// between them) race on the array and produce wrong results; calls on one stream are safe.
#include <cuda.h>

#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

// Size of the built-in split scratch: 16 MiB.
#define PKV_NOALLOC_SCRATCH_BYTES (size_t(16) << 20)

// The scratch itself, one copy per device that loads the library.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace pkv {
namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};  // the context each address was looked up in

// Device address of the scratch on the current device. The array's name is only a host-side
// stand-in in host code, so the address must come from cudaGetSymbolAddress: once per device,
// and again only if the device's context has changed since (a cudaDeviceReset).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(PKV_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(PKV_ECUDA, "device index %d", dev);
  // (no context yet on this thread: the lookup below creates the device's primary context,
  // and the next call, finding that context, looks the address up once more)
  void* const ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess)
      return set_error(PKV_ECUDA, "cudaGetSymbolAddress(decode scratch): %s",
                       cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_decode_noalloc_scratch_bytes(void) { return pkv::kScratchBytes; }

extern "C" int pkv_paged_decode_attention_noalloc(
    const void* q, int32_t dtype_q, int32_t batch, int32_t num_q_heads, const void* k_cache,
    const void* v_cache, const pkv_cache_desc* desc, const int32_t* block_tables,
    int32_t max_pages_per_seq, const int32_t* context_lens, float scale, const float* k_scales,
    const float* v_scales, void* out, void* stream) {
  size_t need = 0;
  if (desc && batch > 0 && num_q_heads > 0 && max_pages_per_seq > 0 && desc->num_kv_heads > 0 &&
      desc->head_dim > 0)
    need = pkv_decode_workspace_size(batch, num_q_heads, desc->num_kv_heads, desc->head_dim,
                                     max_pages_per_seq);
  if (need > pkv::kScratchBytes)
    return pkv::set_error(PKV_EINVAL,
                          "pkv_paged_decode_attention_noalloc: these sizes need %zu bytes of "
                          "split scratch but the built-in scratch holds %zu bytes (16 MiB); use "
                          "pkv_paged_decode_attention with a workspace, or fewer/larger chunks",
                          need, pkv::kScratchBytes);
  void* ws = nullptr;
  if (need > 0) {
    const int st = pkv::scratch_address(&ws);
    if (st != PKV_OK) return st;
    // the per-group chunk counters at the end of the layout must read zero when the decode
    // starts; every call clears them (the rest of the scratch is written before it is read)
    const size_t counters = (size_t)batch * desc->num_kv_heads * sizeof(int);
    const size_t at = need - ((counters + 255) & ~size_t(255));
    const cudaError_t e =
        cudaMemsetAsync(static_cast<char*>(ws) + at, 0, counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return pkv::set_error(PKV_ECUDA, "pkv_paged_decode_attention_noalloc: %s",
                            cudaGetErrorString(e));
  }
  return pkv_paged_decode_attention(q, dtype_q, batch, num_q_heads, k_cache, v_cache, desc,
                                    block_tables, max_pages_per_seq, context_lens, scale, k_scales,
                                    v_scales, out, ws, need > 0 ? pkv::kScratchBytes : 0, stream);
}
