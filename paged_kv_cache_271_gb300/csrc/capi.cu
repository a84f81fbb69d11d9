// C ABI of the library: argument checks, the split-over-pages policy, kernel dispatch, the
// device error word and launch tracing. Every function here returns a pkv_status; argument
// errors are found on the host before anything is launched.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"
#include "pkv_internal.h"

namespace pkv {

// One word per device: kernels OR PKV_DEVERR_* bits into it instead of trapping.
__device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
int* g_err_ptr[kMaxDevices] = {};

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return set_error(PKV_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return set_error(PKV_ECUDA, "device index %d", *dev);
  return PKV_OK;
}

// Device address of the current device's error word (looked up once per device).
int error_word(int** out) {
  int dev = 0;
  int st = current_device(&dev);
  if (st != PKV_OK) return st;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess)
      return set_error(PKV_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return PKV_OK;
}

// ---- tracing --------------------------------------------------------------------------------

struct TraceRec {
  std::string name;
  cudaEvent_t begin, end;
};
std::atomic<bool> g_trace_on{false};
std::mutex g_trace_mu;
std::vector<TraceRec> g_trace;

template <class F>
cudaError_t traced(const char* name, cudaStream_t s, F&& launch) {
  if (!g_trace_on.load(std::memory_order_relaxed)) return launch();
  TraceRec r{name, nullptr, nullptr};
  cudaError_t e = cudaEventCreate(&r.begin);
  if (e == cudaSuccess) e = cudaEventCreate(&r.end);
  if (e != cudaSuccess) return e;
  cudaEventRecord(r.begin, s);
  e = launch();
  cudaEventRecord(r.end, s);
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.push_back(r);
  return e;
}

}  // namespace

void* current_context() {
  using CtxGetCurrent = CUresult (*)(CUcontext*);
  static const CtxGetCurrent fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrent>(f);
  }();
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

int bind_context(const char* who) {
  if (current_context()) return PKV_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);  // initialises the primary context, current
  if (e != cudaSuccess)
    return set_error(PKV_ECUDA, "%s: no context for device %d: %s", who, dev,
                     cudaGetErrorString(e));
  return PKV_OK;
}

cudaError_t traced_copy(const char* name, void* dst, const void* src, size_t bytes,
                        cudaMemcpyKind kind, cudaStream_t s) {
  return traced(name, s, [&] { return cudaMemcpyAsync(dst, src, bytes, kind, s); });
}

namespace {

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return PKV_OK;
  return set_error(PKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int> g_chunk_override{0};
// Calls whose sequences split into at most this many chunks merge them in the decode kernel
// (0: always the combine kernel, the default -- measured faster on every workload tried).
std::atomic<int> g_merge_in_place_max{0};
std::atomic<int> g_kernel_choice{0};  // 0 automatic, 1 CUDA cores, 2 tensor cores
// 0: prefix kernel, then own-page decode; 1: the own-page decode overlaps the prefix kernel and
// folds its partials in; 2: overlaps it and leaves the fold to the combine kernel
std::atomic<int> g_cascade_overlap{2};
std::atomic<int> g_warp_units{1};     // 1: one warp per request for short single-chunk runs
// 0: automatic -- the split measured fastest for the call's shape when one has been recorded
// (autotuning), else chunks; 1: chunks only; 2: the balanced split (decode_flat.cu) wherever it
// applies; 3, 4: chunks 1.5 or 2 times the automatic length wherever they apply
std::atomic<int> g_split_mode{0};

// Autotuning of the split: the first call of a shape (while on, and not during stream capture)
// times both splits and records the faster. Events for the timing are made when it is turned
// on, on that device, so that decode calls create nothing.
constexpr int kTuneReps = 5;
constexpr int kTuneKinds = 4;  // chunks, balanced, chunks 1.5x and 2x longer
struct SplitKey {
  int v[11];
  bool operator<(const SplitKey& o) const {
    return std::lexicographical_compare(v, v + 11, o.v, o.v + 11);
  }
};
std::mutex g_tune_mu;      // the recorded choices
std::mutex g_tune_run_mu;  // the timing runs and their events (one shape timed at a time)
std::map<SplitKey, int> g_tuned;  // the kind measured fastest (decode_impl's run)
std::atomic<int> g_autotune{0};
std::atomic<int> g_tune_dev{-1};
cudaEvent_t g_tune_ev[kTuneKinds * kTuneReps][2];

// ---- TMA tensor maps of the pools (for the tensor-core decode) -------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct MapEntry {
  int dev;
  const void* base;
  long long rows;
  int head_dim;
  int dtype;
  int want;  // the rank asked for
  int rank;  // the rank encoded
  CUtensorMap map;
};
std::mutex g_map_mu;
std::vector<MapEntry> g_maps;
EncodeTiledFn g_encode = nullptr;

// The TMA view of a pool, encoded once per (device, pool, shape). A row of 128 bytes (FP8,
// INT8 at head_dim 128) is a 2-D tensor [num_pages * h_kv * 16 rows][128 bytes], one
// (page, KV head) tile per box of 16 rows. A bf16 row of 256 bytes is a 3-D tensor
// [2 halves][rows][64 elements] (halves 128 bytes apart, rows 256 bytes apart), so that one box
// of 2 x 16 x 64 moves a whole (page, KV head) tile into shared memory as two 128-byte-swizzled
// blocks of 16 rows, the first half of every row before the second (the layout the kernels
// read); *rank receives 2 or 3. force_2d asks for the 2-D view of a bf16 pool too (two boxes
// of 16 rows x 64 elements per tile).
int pool_tensor_map(const void* base, const pkv_cache_desc* d, CUtensorMap* out, int* rank,
                    bool force_2d = false) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return set_error(PKV_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  const long long rows = (long long)d->num_pages * d->num_kv_heads * d->page_size;
  const int eb = d->cache_dtype == PKV_BF16 ? 2 : 1;
  const int want_rank = d->head_dim * eb == 256 && !force_2d ? 3 : 2;
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (auto& e : g_maps)
    if (e.dev == dev && e.base == base && e.rows == rows && e.head_dim == d->head_dim &&
        e.dtype == d->cache_dtype && e.want == want_rank) {
      *out = e.map;
      *rank = e.rank;
      return PKV_OK;
    }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    ce = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                          &q);
    if (ce != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return set_error(PKV_ECUDA, "cuTensorMapEncodeTiled is not available");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  // (the encoder needs a current context; a new host thread may not have one yet)
  const int bst = bind_context("pool tensor map");
  if (bst != PKV_OK) return bst;
  MapEntry e{};
  e.dev = dev;
  e.base = base;
  e.rows = rows;
  e.head_dim = d->head_dim;
  e.dtype = d->cache_dtype;
  e.want = want_rank;
  const CUtensorMapDataType dt =
      eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r;
  if (want_rank == 3) {
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
    const cuuint64_t strides[2] = {256, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)d->page_size, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    r = g_encode(&e.map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    e.rank = 3;
    if (r != CUDA_SUCCESS) e.rank = 2;  // not accepted: two 2-D boxes per tile instead
  }
  if (want_rank == 2 || e.rank == 2) {
    const cuuint64_t dims[2] = {(cuuint64_t)d->head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d->head_dim * eb};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)d->page_size};
    const cuuint32_t estr[2] = {1, 1};
    r = g_encode(&e.map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    e.rank = 2;
  }
  if (r != CUDA_SUCCESS) return set_error(PKV_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  if (g_maps.size() >= 256) g_maps.clear();  // callers keep few pools; drop stale entries
  g_maps.push_back(e);
  *out = e.map;
  *rank = e.rank;
  return PKV_OK;
}

// Largest chunk (pages per CTA); each sequence is split into the fewest near-equal chunks no
// larger than this (64 or 32 pages keep the partials near 1 % of the KV bytes); one chunk
// when every sequence fits in one.
int chunk_pages_for(int batch, int h_kv, int max_pages) {
  const int ov = g_chunk_override.load();
  if (ov > 0) return ov;
  // 64-page chunks when they still give ~3000 CTA slots, else 32 (measured on the
  // Llama-3-8B batch-64, 70B long-context, prefix-sharing and FP8 batch-256 workloads);
  // smaller while there would be fewer than ~1024 slots.
  const long long units = (long long)batch * h_kv;
  int chunk = units * ((max_pages + 63) / 64) >= 3000 ? 64 : 32;
  while (chunk > 8 && units * ((max_pages + chunk - 1) / chunk) < 1024) chunk /= 2;
  if (max_pages <= chunk) chunk = max_pages < 1 ? 1 : max_pages;
  return chunk;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: acc [batch][h_q][slots][d] and (max, sum) [batch][h_q][slots][2] floats, then one
// counter per (request, KV head) for the in-place merge; 256-byte aligned regions.
// The balanced split's partials take a region of their own after those (before the counters):
// [G][cap][head_dim] values, [G][cap][2] (max, sum) and [batch + 1] per-request page offsets,
// cap = batch * h_kv + warps, for at most
// a wave of four 4-warp CTAs on each of 152 SMs and no more warps than a quarter of the pages
// the table can hold. It is part of the layout of a plain decode call with an automatic chunk
// size, more than one chunk slot, batch <= kFlatMaxBatch and room for one CTA.
constexpr int kFlatBudgetWarps = 152 * 4 * kFlatWarpsPerCta;

int flat_warps_for(int batch, int h_kv, int max_pages) {
  const long long w = std::min<long long>(kFlatBudgetWarps, (long long)batch * h_kv * max_pages / 4);
  return (int)(w / kFlatWarpsPerCta * kFlatWarpsPerCta);
}

bool flat_region_for(int batch, int h_kv, int max_pages, bool cascade, int slots) {
  return !cascade && slots > 1 && batch <= kFlatMaxBatch && g_chunk_override.load() == 0 &&
         flat_warps_for(batch, h_kv, max_pages) >= kFlatWarpsPerCta;
}

size_t flat_cap_for(int batch, int h_kv, int max_pages) {
  return (size_t)batch * h_kv + flat_warps_for(batch, h_kv, max_pages);
}

size_t workspace_bytes_for(int batch, int h_q, int h_kv, int head_dim, int slots,
                           size_t flat_cap = 0) {
  const size_t rows = (size_t)batch * h_q * slots, frows = flat_cap * (h_q / h_kv);
  return align256(rows * head_dim * sizeof(float)) + align256(rows * 2 * sizeof(float)) +
         (flat_cap ? align256(frows * head_dim * sizeof(float)) +
                         align256(frows * 2 * sizeof(float)) +
                         align256(((size_t)batch + 1) * sizeof(int))
                   : 0) +
         align256((size_t)batch * h_kv * sizeof(int));
}

std::atomic<int> g_prefix_chunk_override{0};

std::atomic<int> g_prefix_kernel{0};  // 0 automatic (tcgen05), 1 mma.sync, 2 tcgen05
bool prefix_on_tcgen05() { return g_prefix_kernel.load() != 1; }

// Pages per CTA of the cascade prefix kernel: the shared pages of each (group, KV head, rows
// of a CTA) are cut into as many chunks as keep the launch within one wave of resident CTAs
// (tcgen05: 128 rows per CTA, one CTA per SM, chunks of at least one 4-page tile;
// mma.sync: 64 rows, three CTAs per SM, at least 2 pages); a chunk of at most the whole prefix.
int prefix_chunk_pages_for(int n_groups, int h_kv, int group, int max_members, int max_prefix) {
  const int ov = g_prefix_chunk_override.load();
  if (ov > 0) return ov;
  if (max_prefix < 1) return 1;
  const bool tc = prefix_on_tcgen05();
  const int rows = tc ? kCascadeTcRows : kCascadeRows;
  // with the fold left to the combine, the tcgen05 prefix kernel takes about half the SMs and
  // the own-page decode runs on the rest meanwhile (prefix sharing, batch 128: two chunks,
  // 38.1 us a step, against 41.1 us with the prefix kernel on every SM)
  const int wave = tc ? (g_cascade_overlap.load() == 2 ? kCascadeTcWaveCtas / 2 : kCascadeTcWaveCtas)
                      : kCascadeWaveCtas;
  const int min_pages = tc ? 4 : 2;
  const long long tiles = ((long long)max_members * group + rows - 1) / rows;
  const long long units = (long long)n_groups * h_kv * tiles;
  long long chunks = wave / (units > 0 ? units : 1);
  chunks = std::max(1ll, std::min(chunks, (long long)(max_prefix + min_pages - 1) / min_pages));
  return (int)((max_prefix + chunks - 1) / chunks);
}

// Pages any request of a cascade decode reads itself (the hint, else the table width).
int cascade_own_pages(int max_pages, const pkv_cascade_desc* g) {
  return g->max_own_pages > 0 && g->max_own_pages < max_pages ? g->max_own_pages : max_pages;
}

// Chunk columns of the decode grid and chunk slots of a cascade decode: the prefix chunks
// first, then the requests' own chunks.
void cascade_split(int batch, int h_kv, int h_q, int max_pages, const pkv_cascade_desc* g,
                   int* chunk_pages, int* chunk_grid, int* prefix_chunk_pages, int* slots) {
  const int own = cascade_own_pages(max_pages, g);
  *chunk_pages = chunk_pages_for(batch, h_kv, own);
  *chunk_grid = (own + *chunk_pages - 1) / *chunk_pages;
  *prefix_chunk_pages =
      prefix_chunk_pages_for(g->n_groups, h_kv, h_q / h_kv, g->max_members, g->max_prefix_pages);
  *slots = *chunk_grid + (g->max_prefix_pages + *prefix_chunk_pages - 1) / *prefix_chunk_pages;
}

int check_desc(const pkv_cache_desc* d, const char* who) {
  if (!d) return set_error(PKV_EINVAL, "%s: desc is NULL", who);
  if (d->page_size != 16) return set_error(PKV_EINVAL, "%s: page_size must be 16", who);
  if (d->head_dim != 64 && d->head_dim != 128)
    return set_error(PKV_ESHAPE, "%s: head_dim must be 64 or 128", who);
  if (d->num_pages <= 0 || d->num_kv_heads <= 0)
    return set_error(PKV_ESHAPE, "%s: num_pages and num_kv_heads must be positive", who);
  if (d->cache_dtype != PKV_F32 && d->cache_dtype != PKV_BF16 && d->cache_dtype != PKV_FP8_E4M3 &&
      d->cache_dtype != PKV_INT8)
    return set_error(PKV_EDTYPE, "%s: unknown cache dtype %d", who, d->cache_dtype);
  if ((long long)d->num_pages * d->num_kv_heads * d->page_size >= (1ll << 40))
    return set_error(PKV_ESHAPE, "%s: pool too large", who);
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_decode_set_chunk_pages(int32_t pages) {
  if (pages < 0 || pages > 4096)
    return set_error(PKV_EINVAL, "pkv_decode_set_chunk_pages: %d outside [0, 4096]", pages);
  g_chunk_override.store(pages);
  return PKV_OK;
}

int pkv_decode_set_merge_in_place(int32_t max_chunks) {
  if (max_chunks < 0 || max_chunks > 4096)
    return set_error(PKV_EINVAL, "pkv_decode_set_merge_in_place: %d outside [0, 4096]", max_chunks);
  g_merge_in_place_max.store(max_chunks);
  return PKV_OK;
}

int pkv_decode_set_kernel(int32_t which) {
  if (which < 0 || which > 2)
    return set_error(PKV_EINVAL, "pkv_decode_set_kernel: %d is not 0, 1 or 2", which);
  g_kernel_choice.store(which);
  return PKV_OK;
}

int pkv_decode_set_warp_per_request(int32_t on) {
  if (on != 0 && on != 1)
    return set_error(PKV_EINVAL, "pkv_decode_set_warp_per_request: %d is not 0 or 1", on);
  g_warp_units.store(on);
  return PKV_OK;
}

int pkv_decode_set_split(int32_t mode) {
  if (mode < 0 || mode > 4)
    return set_error(PKV_EINVAL, "pkv_decode_set_split: %d is not in 0..4", mode);
  g_split_mode.store(mode);
  return PKV_OK;
}

int pkv_decode_set_autotune(int32_t on) {
  if (on != 0 && on != 1)
    return set_error(PKV_EINVAL, "pkv_decode_set_autotune: %d is not 0 or 1", on);
  std::lock_guard<std::mutex> run_lk(g_tune_run_mu);  // (no timing run uses the events now)
  std::lock_guard<std::mutex> lk(g_tune_mu);
  if (on) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "pkv_decode_set_autotune");
    if (g_tune_dev != dev) {
      if (g_tune_dev >= 0) {
        int cur = dev;
        cudaSetDevice(g_tune_dev.load());
        for (auto& pr : g_tune_ev) {
          cudaEventDestroy(pr[0]);
          cudaEventDestroy(pr[1]);
        }
        cudaSetDevice(cur);
        g_tune_dev = -1;
      }
      for (auto& pr : g_tune_ev) {
        e = cudaEventCreate(&pr[0]);
        if (e == cudaSuccess) e = cudaEventCreate(&pr[1]);
        if (e != cudaSuccess) return cuda_status(e, "pkv_decode_set_autotune: events");
      }
      g_tune_dev = dev;
    }
  }
  g_autotune.store(on);
  return PKV_OK;
}

int pkv_decode_autotune_reset(void) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tuned.clear();
  return PKV_OK;
}

int pkv_decode_split_choice(int32_t kv_dtype, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t max_pages_per_seq, int32_t window,
                            int32_t sink_tokens, int32_t fused) {
  // (the key as decode_impl forms it; slots follow from the other fields and the chunk policy)
  std::lock_guard<std::mutex> lk(g_tune_mu);
  for (const auto& kv : g_tuned) {
    const int* v = kv.first.v;
    if (v[0] == kv_dtype && v[1] == q_dtype && v[2] == batch && v[3] == num_q_heads &&
        v[4] == num_kv_heads && v[5] == max_pages_per_seq && v[6] == window &&
        v[7] == (window > 0 ? sink_tokens : 0) && v[8] == (fused ? 1 : 0))
      return kv.second;
  }
  return -1;
}

int pkv_cascade_set_overlap(int32_t on) {
  if (on < 0 || on > 2)
    return set_error(PKV_EINVAL, "pkv_cascade_set_overlap: %d is not 0, 1 or 2", on);
  g_cascade_overlap.store(on);
  return PKV_OK;
}

int32_t pkv_decode_chunk_pages(int32_t batch, int32_t num_kv_heads, int32_t max_pages_per_seq) {
  return chunk_pages_for(batch, num_kv_heads, max_pages_per_seq);
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_pages_per_seq) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_pages_per_seq <= 0)
    return 0;
  const int chunk = chunk_pages_for(batch, num_kv_heads, max_pages_per_seq);
  const int slots = (max_pages_per_seq + chunk - 1) / chunk;
  if (slots <= 1) return 0;
  const bool flat = flat_region_for(batch, num_kv_heads, max_pages_per_seq, false, slots);
  return workspace_bytes_for(batch, num_q_heads, num_kv_heads, head_dim, slots,
                             flat ? flat_cap_for(batch, num_kv_heads, max_pages_per_seq) : 0);
}

int32_t pkv_cascade_prefix_chunk_pages(int32_t num_kv_heads, int32_t num_q_heads,
                                       const pkv_cascade_desc* groups) {
  if (!groups || groups->n_groups <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
      groups->max_prefix_pages <= 0 || groups->max_members <= 0)
    return 0;
  return prefix_chunk_pages_for(groups->n_groups, num_kv_heads, num_q_heads / num_kv_heads,
                                groups->max_members, groups->max_prefix_pages);
}

size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_pages_per_seq,
                                  const pkv_cascade_desc* groups) {
  if (!groups || groups->n_groups <= 0)
    return pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                     max_pages_per_seq);
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_pages_per_seq <= 0 || groups->max_prefix_pages <= 0 || groups->max_members <= 0)
    return 0;
  int chunk, grid, pchunk, slots;
  cascade_split(batch, num_kv_heads, num_q_heads, max_pages_per_seq, groups, &chunk, &grid,
                &pchunk, &slots);
  return workspace_bytes_for(batch, num_q_heads, num_kv_heads, head_dim, slots);
}

static int decode_impl(const char* who, const void* q, int32_t dtype_q, int32_t batch,
                       int32_t num_q_heads, const void* k_cache, const void* v_cache,
                       const pkv_cache_desc* desc, const int32_t* block_tables,
                       int32_t max_pages_per_seq, const int32_t* context_lens, float scale,
                       const float* k_scales, const float* v_scales, void* out, void* workspace,
                       size_t workspace_bytes, const void* k_new, const void* v_new,
                       int32_t dtype_new, int32_t sink_tokens, int32_t window,
                       const pkv_cascade_desc* groups, void* stream) {
  int st = check_desc(desc, who);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0)
    return set_error(PKV_EINVAL, "%s: bad batch, head count or table width", who);
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return set_error(PKV_EINVAL, "%s: null pointer", who);
  const int h_kv = desc->num_kv_heads, D = desc->head_dim;
  if (num_q_heads % h_kv != 0)
    return set_error(PKV_ESHAPE, "%s: num_q_heads %% num_kv_heads != 0", who);
  const int G = num_q_heads / h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return set_error(PKV_ESHAPE, "%s: group size %d not in {1,2,4,8,16}", who, G);
  const int kv = desc->cache_dtype;
  if (dtype_q != PKV_F32 && dtype_q != PKV_BF16)
    return set_error(PKV_EDTYPE, "%s: q dtype must be F32 or BF16", who);
  if ((kv == PKV_F32 && dtype_q != PKV_F32) || (kv == PKV_BF16 && dtype_q != PKV_BF16))
    return set_error(PKV_EDTYPE, "%s: q dtype must match an F32/BF16 cache", who);
  const bool coded = kv == PKV_FP8_E4M3 || kv == PKV_INT8;
  if (coded && (!k_scales || !v_scales))
    return set_error(PKV_EINVAL, "%s: FP8/INT8 cache needs k_scales and v_scales", who);
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return set_error(PKV_EALIGN, "%s: pools must be 16-byte aligned", who);
  if (!(scale == scale)) return set_error(PKV_EINVAL, "%s: scale is NaN", who);
  if (window < 0 || sink_tokens < 0 || (window == 0 && sink_tokens != 0))
    return set_error(PKV_EINVAL, "%s: window and sink_tokens must be >= 0; sinks need a window",
                     who);
  if (h_kv > 65535 || batch > 65535)
    return set_error(PKV_ESHAPE, "%s: batch and kv heads must be <= 65535", who);

  DecodeArgs a{};
  a.q = q;
  a.out = out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.batch = batch;
  a.h_q = num_q_heads;
  a.h_kv = h_kv;
  a.num_pages = desc->num_pages;
  a.max_pages = max_pages_per_seq;
  a.chunk_pages = chunk_pages_for(batch, h_kv, max_pages_per_seq);
  a.n_chunk_slots = (max_pages_per_seq + a.chunk_pages - 1) / a.chunk_pages;
  int walk_pages = max_pages_per_seq;  // the most pages a request can walk
  if (window > 0) {
    // a windowed request walks at most its sink pages, the window's pages and one boundary
    // page: the chunks are sized for that run, not for the table width (while the partials
    // still fit the workspace sized for the table width)
    const long long run =
        ((long long)sink_tokens + desc->page_size - 1) / desc->page_size +
        ((long long)window + desc->page_size - 1) / desc->page_size + 1;
    const int walk = (int)std::min<long long>(max_pages_per_seq, run);
    int chunk = chunk_pages_for(batch, h_kv, walk);
    while ((walk + chunk - 1) / chunk > a.n_chunk_slots) chunk *= 2;
    a.chunk_pages = chunk;
    a.n_chunk_slots = (walk + chunk - 1) / chunk;
    walk_pages = walk;
  }
  a.chunk_grid = a.n_chunk_slots;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.window = window;
  a.sink = window > 0 ? sink_tokens : 0;
  const bool cascade = groups != nullptr && groups->n_groups > 0;
  CascadeArgs ca{};
  if (cascade) {
    if (!groups->group_of || !groups->prefix_pages || !groups->group_offsets ||
        !groups->group_members)
      return set_error(PKV_EINVAL, "%s: cascade groups with a null array", who);
    if (groups->max_members < 1 || groups->max_members > batch || groups->max_prefix_pages < 1 ||
        groups->max_prefix_pages > max_pages_per_seq || groups->n_groups > batch)
      return set_error(PKV_EINVAL, "%s: cascade bounds outside [1, batch] members, [1, table "
                       "width] prefix pages, <= batch groups", who);
    if (window != 0)
      return set_error(PKV_EINVAL, "%s: a cascade decode takes no window", who);
    if (kv != PKV_BF16 || D != 128 || !aligned16(q) ||
        (long long)desc->num_pages * h_kv * desc->page_size >= (1ll << 31))
      return set_error(PKV_EDTYPE, "%s: the cascade decode needs a bf16 cache and queries, "
                       "head_dim 128, a 16-byte aligned q and fewer than 2^31 pool rows", who);
    if ((long long)groups->n_groups * h_kv > 65535)
      return set_error(PKV_ESHAPE, "%s: groups * kv heads must be <= 65535", who);
    a.group_of = groups->group_of;
    a.prefix_pages = groups->prefix_pages;
    a.own_start = groups->own_start;
    a.n_groups = groups->n_groups;
    a.max_prefix_pages = groups->max_prefix_pages;
    cascade_split(batch, h_kv, num_q_heads, max_pages_per_seq, groups, &a.chunk_pages,
                  &a.chunk_grid, &a.prefix_chunk_pages, &a.n_chunk_slots);
    ca.group_offsets = groups->group_offsets;
    ca.group_members = groups->group_members;
    ca.max_members = groups->max_members;
    ca.prefix_ids = groups->prefix_page_ids;
    ca.ids_stride = groups->max_prefix_pages;
  }
  if (a.n_chunk_slots > 65535) return set_error(PKV_ESHAPE, "%s: too many chunks", who);
  bool flat_region = false;  // the workspace holds the balanced split's partials too
  float* flat_acc = nullptr;
  float* flat_ml = nullptr;
  if (a.n_chunk_slots > 1) {
    flat_region = flat_region_for(batch, h_kv, max_pages_per_seq, cascade, a.n_chunk_slots);
    const size_t fcap = flat_region ? flat_cap_for(batch, h_kv, max_pages_per_seq) : 0;
    const size_t need = workspace_bytes_for(batch, num_q_heads, h_kv, D, a.n_chunk_slots, fcap);
    if (!workspace || workspace_bytes < need)
      return set_error(PKV_EINVAL, "%s: workspace of %zu bytes needed, %zu given", who, need,
                       workspace_bytes);
    if (!aligned16(workspace)) return set_error(PKV_EALIGN, "%s: workspace alignment", who);
    const size_t rows = (size_t)batch * num_q_heads * a.n_chunk_slots;
    char* ws = static_cast<char*>(workspace);
    size_t off = 0;
    a.ws_acc = reinterpret_cast<float*>(ws);
    off += align256(rows * D * sizeof(float));
    a.ws_ml = reinterpret_cast<float*>(ws + off);
    off += align256(rows * 2 * sizeof(float));
    if (flat_region) {
      const size_t frows = fcap * G;
      flat_acc = reinterpret_cast<float*>(ws + off);
      off += align256(frows * D * sizeof(float));
      flat_ml = reinterpret_cast<float*>(ws + off);
      off += align256(frows * 2 * sizeof(float));
      a.flat_pre = reinterpret_cast<int*>(ws + off);
      off += align256(((size_t)batch + 1) * sizeof(int));
    }
    a.counters = reinterpret_cast<int*>(ws + off);
    // few chunks per sequence: the last CTA of each group merges them (no combine kernel).
    // A cascade decode that folds in the own-page kernel (overlap modes 0 and 1) always merges
    // there: a request's one own chunk folds in its prefix partials, several own chunks merge
    // in place; with the fold left to the combine (mode 2) this is undone below.
    a.merge_in_place = cascade || a.n_chunk_slots <= g_merge_in_place_max.load() ? 1 : 0;
  }
  if (k_new) {
    if (!v_new) return set_error(PKV_EINVAL, "%s: v_new is NULL", who);
    if (coded) {
      if (dtype_new != PKV_F32 && dtype_new != PKV_BF16)
        return set_error(PKV_EDTYPE, "%s: FP8/INT8 cache takes F32 or BF16 new rows", who);
    } else if (dtype_new != kv) {
      return set_error(PKV_EDTYPE, "%s: new rows must have the cache dtype", who);
    }
    if (!aligned16(k_new) || !aligned16(v_new))
      return set_error(PKV_EALIGN, "%s: new rows must be 16-byte aligned", who);
    a.k_new = k_new;
    a.v_new = v_new;
    a.new_dtype = dtype_new;
  }
  const int choice = g_kernel_choice.load();
  const bool mma_ok = kv != PKV_F32 && D == 128 && aligned16(q) &&
                      (long long)desc->num_pages * h_kv * desc->page_size < (1ll << 31);
  if (choice == 2 && !mma_ok)
    return set_error(PKV_EINVAL, "%s: the tensor-core decode needs a bf16 or FP8 cache, head_dim "
                     "128, a 16-byte aligned q and fewer than 2^31 pool rows", who);
  const bool use_mma = mma_ok && choice != 1;
  // every request in one chunk of at most 16 pages: one warp per request (short runs would
  // leave a CTA's four warps with a page or two each)
  // (one chunk column: no request splits, so no merge of chunk partials can arise)
  a.warp_units = use_mma && a.chunk_grid == 1 && a.chunk_pages <= 16 && g_warp_units.load() != 0;
  // Splits of a plain call on the tensor-core kernel whose partials go to a combine kernel:
  // the chunks (kind 0), the balanced split (kind 1: one wave of CTAs, equal shares of the
  // (request, KV head, page) stream per warp, decode_flat.cu; its partials in the workspace's
  // region for them), and, when the chunk size is automatic, chunks 1.5 and 2 times longer
  // (kinds 2 and 3: fewer CTAs and waves; their partials fit the slots of the automatic size).
  const int split_mode = g_split_mode.load();
  const bool flat_applies = use_mma && flat_region && !a.merge_in_place && split_mode != 1;
  const bool longer_applies = use_mma && !cascade && a.n_chunk_slots > 1 && !a.merge_in_place &&
                              g_chunk_override.load() == 0 && split_mode != 1 && split_mode != 2;
  int flat_ctas = 0, flat_cap = 0;  // the balanced split's launch, worked out when it may run
  auto flat_plan = [&]() {
    const long long cap = (long long)flat_cap_for(batch, h_kv, max_pages_per_seq);
    int wave = 0;
    if (cap < (1ll << 31) && decode_flat_wave(a, kv, dtype_q, G, &wave) == cudaSuccess) {
      flat_ctas = std::min(flat_warps_for(batch, h_kv, max_pages_per_seq) / kFlatWarpsPerCta,
                           wave);
      flat_cap = (int)cap;
    }
    return flat_ctas > 0;
  };
  a.prefix_dep = cascade && use_mma && g_cascade_overlap.load() != 0 ? 1 : 0;
  a.defer_fold = a.prefix_dep && g_cascade_overlap.load() == 2 ? 1 : 0;
  if (a.defer_fold) a.merge_in_place = 0;  // every member's chunks go to the combine
  CUtensorMap tk, tv;
  if (use_mma || cascade) {
    int rk = 2, rv = 2;
    st = pool_tensor_map(k_cache, desc, &tk, &rk);
    if (st == PKV_OK) st = pool_tensor_map(v_cache, desc, &tv, &rv);
    if (st == PKV_OK && rk != rv) st = set_error(PKV_ECUDA, "%s: pool tensor maps differ", who);
    a.tma_rank = rk;
    if (st != PKV_OK) return st;
  }
  st = error_word(&a.err);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (cascade) {
    CUtensorMap tk2;
    if (prefix_on_tcgen05()) {  // its K operand needs 2-D boxes (see cascade_prefix_tc.cu)
      int r2 = 0;
      st = pool_tensor_map(k_cache, desc, &tk2, &r2, true);
      if (st != PKV_OK) return st;
    }
    e = traced("cascade_prefix", s, [&] {
      return prefix_on_tcgen05() ? launch_cascade_prefix_tc(a, ca, G, &tk2, &tv, s)
                                 : launch_cascade_prefix(a, ca, G, &tk, &tv, s);
    });
    st = cuda_status(e, "cascade_prefix launch");
    if (st != PKV_OK) return st;
  }
  // the decode (and its combine) with split kind 0..3 (above)
  // (ev: events recorded around the decode kernel, for autotuning)
  auto run = [&](int kind, cudaEvent_t* ev = nullptr) {
    DecodeArgs af = a;  // the balanced split's arguments: partials in their own region
    af.ws_acc = flat_acc;
    af.ws_ml = flat_ml;
    DecodeArgs ac = a;  // the chunks' arguments (longer chunks: the same partial slots)
    if (kind >= 2) {
      ac.chunk_pages = std::min(4096, kind == 2 ? a.chunk_pages * 3 / 2 : a.chunk_pages * 2);
      ac.chunk_grid = (walk_pages + ac.chunk_pages - 1) / ac.chunk_pages;
    }
    if (ev) cudaEventRecord(ev[0], s);
    cudaError_t err = traced("paged_decode", s, [&] {
      if (kind == 1)
        return launch_decode_flat(af, kv, dtype_q, G, flat_ctas, flat_cap, &tk, &tv, s);
      if (use_mma) return launch_decode_mma(ac, kv, dtype_q, G, &tk, &tv, s);
      if (kv == PKV_F32) return launch_decode_f32(a, dtype_q, D, G, s);
      if (kv == PKV_BF16) return launch_decode_bf16(a, dtype_q, D, G, s);
      if (kv == PKV_INT8) return launch_decode_int8(a, dtype_q, D, G, s);
      return launch_decode_fp8(a, dtype_q, D, G, s);
    });
    if (ev) cudaEventRecord(ev[1], s);
    int rs = cuda_status(err, "paged_decode launch");
    if (rs != PKV_OK) return rs;
    if (kind == 1) {
      err = traced("decode_combine", s, [&] {
        return launch_decode_flat_combine(af, kv, dtype_q, G, flat_ctas, flat_cap, s);
      });
      rs = cuda_status(err, "decode_combine launch");
    } else if (a.n_chunk_slots > 1 && !a.merge_in_place) {
      err = traced("decode_combine", s, [&] { return launch_decode_combine(ac, dtype_q, D, s); });
      rs = cuda_status(err, "decode_combine launch");
    }
    return rs;
  };
  if (split_mode == 2) return run(flat_applies && flat_plan() ? 1 : 0);
  if (split_mode >= 3) return run(longer_applies ? split_mode - 1 : 0);
  if (!flat_applies && !longer_applies) return run(0);
  // a recorded kind that still applies (a balanced one needs its launch worked out)
  auto usable = [&](int kind) {
    if (kind == 1) return flat_applies && flat_plan() ? 1 : 0;
    return kind >= 2 && !longer_applies ? 0 : kind;
  };
  // automatic: the recorded choice for this shape, else (autotuning, not capturing) measure
  const SplitKey key{{kv, dtype_q, batch, num_q_heads, h_kv, max_pages_per_seq, window, a.sink,
                      k_new ? 1 : 0, a.n_chunk_slots, 0}};
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    auto it = g_tuned.find(key);
    if (it != g_tuned.end()) return run(usable(it->second));
  }
  int dev = -1;
  cudaStreamCaptureStatus cap_st = cudaStreamCaptureStatusNone;
  if (!g_autotune.load() || cudaGetDevice(&dev) != cudaSuccess || dev != g_tune_dev ||
      cudaStreamIsCapturing(s, &cap_st) != cudaSuccess || cap_st != cudaStreamCaptureStatusNone)
    return run(0);
  // every kind that applies, in turn, kTuneReps times each; the one whose decode kernel took
  // the least time over its runs is recorded and gives this call's result (the appended row is
  // written again each run). The combine is left out of the timing: in a step replayed from a
  // graph it starts beside the decode's last CTAs, and its own work is small and similar.
  int kinds[kTuneKinds], n_kinds = 0;
  kinds[n_kinds++] = 0;
  if (flat_applies && flat_plan()) kinds[n_kinds++] = 1;
  if (longer_applies) {
    kinds[n_kinds++] = 2;
    kinds[n_kinds++] = 3;
  }
  if (n_kinds == 1) return run(0);
  float best[kTuneKinds];
  int pick = 0;
  {
    std::lock_guard<std::mutex> run_lk(g_tune_run_mu);
    {  // another thread may have timed this shape meanwhile
      std::lock_guard<std::mutex> lk(g_tune_mu);
      auto it = g_tuned.find(key);
      if (it != g_tuned.end()) return run(usable(it->second));
    }
    for (int rep = 0; rep < kTuneReps && st == PKV_OK; ++rep)
      for (int f = 0; f < n_kinds && st == PKV_OK; ++f)
        st = run(kinds[f], g_tune_ev[kTuneKinds * rep + f]);
    if (st != PKV_OK) return st;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e, "decode split autotune");
    for (int f = 0; f < n_kinds; ++f) {
      best[f] = 1e30f;
      for (int rep = 0; rep < kTuneReps; ++rep) {
        float ms = 0.f;
        cudaEvent_t* ev = g_tune_ev[kTuneKinds * rep + f];
        if (cudaEventElapsedTime(&ms, ev[0], ev[1]) == cudaSuccess) best[f] = std::min(best[f], ms);
      }
      if (best[f] < best[pick]) pick = f;
    }
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tuned[key] = kinds[pick];
  }
  return run(kinds[pick]);
}

int pkv_paged_decode_attention(const void* q, int32_t dtype_q, int32_t batch,
                               int32_t num_q_heads, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* desc, const int32_t* block_tables,
                               int32_t max_pages_per_seq, const int32_t* context_lens,
                               float scale, const float* k_scales, const float* v_scales,
                               void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl("pkv_paged_decode_attention", q, dtype_q, batch, num_q_heads, k_cache,
                     v_cache, desc, block_tables, max_pages_per_seq, context_lens, scale,
                     k_scales, v_scales, out, workspace, workspace_bytes, nullptr, nullptr, 0, 0,
                     0, nullptr, stream);
}

int pkv_paged_decode_attention_window(const void* q, int32_t dtype_q, int32_t batch,
                                      int32_t num_q_heads, const void* k_cache,
                                      const void* v_cache, const pkv_cache_desc* desc,
                                      const int32_t* block_tables, int32_t max_pages_per_seq,
                                      const int32_t* context_lens, float scale,
                                      const float* k_scales, const float* v_scales,
                                      int32_t sink_tokens, int32_t window, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl("pkv_paged_decode_attention_window", q, dtype_q, batch, num_q_heads,
                     k_cache, v_cache, desc, block_tables, max_pages_per_seq, context_lens, scale,
                     k_scales, v_scales, out, workspace, workspace_bytes, nullptr, nullptr, 0,
                     sink_tokens, window, nullptr, stream);
}

int pkv_paged_decode_step(const void* q, int32_t dtype_q, int32_t batch, int32_t num_q_heads,
                          const void* k_new, const void* v_new, int32_t dtype_new,
                          void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                          const int32_t* block_tables, int32_t max_pages_per_seq,
                          const int32_t* context_lens, float scale, const float* k_scales,
                          const float* v_scales, void* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!k_new && batch != 0)  // (an empty batch may pass null pointers)
    return set_error(PKV_EINVAL, "pkv_paged_decode_step: k_new is NULL");
  return decode_impl("pkv_paged_decode_step", q, dtype_q, batch, num_q_heads, k_cache, v_cache,
                     desc, block_tables, max_pages_per_seq, context_lens, scale, k_scales,
                     v_scales, out, workspace, workspace_bytes, k_new, v_new, dtype_new, 0, 0,
                     nullptr, stream);
}

int pkv_paged_decode_step_window(const void* q, int32_t dtype_q, int32_t batch,
                                 int32_t num_q_heads, const void* k_new, const void* v_new,
                                 int32_t dtype_new, void* k_cache, void* v_cache,
                                 const pkv_cache_desc* desc, const int32_t* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* context_lens,
                                 float scale, const float* k_scales, const float* v_scales,
                                 int32_t sink_tokens, int32_t window, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!k_new && batch != 0)
    return set_error(PKV_EINVAL, "pkv_paged_decode_step_window: k_new is NULL");
  return decode_impl("pkv_paged_decode_step_window", q, dtype_q, batch, num_q_heads, k_cache,
                     v_cache, desc, block_tables, max_pages_per_seq, context_lens, scale,
                     k_scales, v_scales, out, workspace, workspace_bytes, k_new, v_new,
                     dtype_new, sink_tokens, window, nullptr, stream);
}



int pkv_packed_step_layout(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t max_pages_per_seq, int32_t dtype_q,
                           int32_t dtype_new, size_t* offsets, size_t* total_bytes) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_pages_per_seq <= 0 || !offsets || !total_bytes)
    return set_error(PKV_EINVAL, "pkv_packed_step_layout: bad argument");
  auto esize = [](int dt) { return dt == PKV_F32 ? 4 : dt == PKV_BF16 ? 2 : 0; };
  if (!esize(dtype_q) || !esize(dtype_new))
    return set_error(PKV_EDTYPE, "pkv_packed_step_layout: q and new rows are F32 or BF16");
  const size_t sz[5] = {(size_t)batch * num_q_heads * head_dim * esize(dtype_q),
                        (size_t)batch * num_kv_heads * head_dim * esize(dtype_new),
                        (size_t)batch * num_kv_heads * head_dim * esize(dtype_new),
                        (size_t)batch * max_pages_per_seq * 4, (size_t)batch * 4};
  size_t off = 0;
  for (int i = 0; i < 5; ++i) {
    offsets[i] = off;
    off += align256(sz[i]);
  }
  *total_bytes = off;
  return PKV_OK;
}

int pkv_paged_decode_step_packed(const void* host_in, void* dev_in, int32_t batch,
                                 int32_t num_q_heads, int32_t dtype_q, int32_t dtype_new,
                                 void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                 int32_t max_pages_per_seq, float scale, const float* k_scales,
                                 const float* v_scales, int32_t sink_tokens, int32_t window,
                                 void* out_dev, void* out_host, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const char* who = "pkv_paged_decode_step_packed";
  int st = check_desc(desc, who);
  if (st != PKV_OK) return st;
  size_t off[5], total = 0;
  st = pkv_packed_step_layout(batch, num_q_heads, desc->num_kv_heads, desc->head_dim,
                              max_pages_per_seq, dtype_q, dtype_new, off, &total);
  if (st != PKV_OK) return st;
  if (batch == 0) return PKV_OK;  // (an empty batch may pass null buffers)
  if (!host_in || !dev_in || !out_dev || !out_host)
    return set_error(PKV_EINVAL, "%s: null pointer", who);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced_copy("h2d_copy", dev_in, host_in, total, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_status(e, "packed step inputs copy");
  char* d = static_cast<char*>(dev_in);
  st = decode_impl(who, d + off[0], dtype_q, batch, num_q_heads, k_cache, v_cache, desc,
                   reinterpret_cast<const int32_t*>(d + off[3]), max_pages_per_seq,
                   reinterpret_cast<const int32_t*>(d + off[4]), scale, k_scales, v_scales,
                   out_dev, workspace, workspace_bytes, d + off[1], d + off[2], dtype_new,
                   sink_tokens, window, nullptr, stream);
  if (st != PKV_OK) return st;
  const size_t out_bytes =
      (size_t)batch * num_q_heads * desc->head_dim * (dtype_q == PKV_F32 ? 4 : 2);
  e = traced_copy("d2h_copy", out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, s);
  return cuda_status(e, "packed step output copy");
}

int pkv_cascade_decode_attention(const void* q, int32_t dtype_q, int32_t batch,
                                 int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                 const pkv_cache_desc* desc, const int32_t* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* context_lens,
                                 float scale, const pkv_cascade_desc* groups, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl("pkv_cascade_decode_attention", q, dtype_q, batch, num_q_heads, k_cache,
                     v_cache, desc, block_tables, max_pages_per_seq, context_lens, scale, nullptr,
                     nullptr, out, workspace, workspace_bytes, nullptr, nullptr, 0, 0, 0, groups,
                     stream);
}

int pkv_cascade_decode_step(const void* q, int32_t dtype_q, int32_t batch, int32_t num_q_heads,
                            const void* k_new, const void* v_new, int32_t dtype_new,
                            void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                            const int32_t* block_tables, int32_t max_pages_per_seq,
                            const int32_t* context_lens, float scale,
                            const pkv_cascade_desc* groups, void* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!k_new && batch != 0)
    return set_error(PKV_EINVAL, "pkv_cascade_decode_step: k_new is NULL");
  return decode_impl("pkv_cascade_decode_step", q, dtype_q, batch, num_q_heads, k_cache,
                     v_cache, desc, block_tables, max_pages_per_seq, context_lens, scale, nullptr,
                     nullptr, out, workspace, workspace_bytes, k_new, v_new, dtype_new, 0, 0,
                     groups, stream);
}

int pkv_cascade_set_prefix_kernel(int32_t which) {
  if (which < 0 || which > 2)
    return set_error(PKV_EINVAL, "pkv_cascade_set_prefix_kernel: %d is not 0, 1 or 2", which);
  g_prefix_kernel.store(which);
  return PKV_OK;
}

int pkv_cascade_set_prefix_chunk_pages(int32_t pages) {
  if (pages < 0 || pages > 4096)
    return set_error(PKV_EINVAL, "pkv_cascade_set_prefix_chunk_pages: %d outside [0, 4096]",
                     pages);
  g_prefix_chunk_override.store(pages);
  return PKV_OK;
}

int pkv_kv_append(const void* k_new, const void* v_new, int32_t dtype_new, int32_t num_tokens,
                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                  const pkv_cache_desc* desc, const float* k_scales, const float* v_scales,
                  void* stream) {
  const char* who = "pkv_kv_append";
  int st = check_desc(desc, who);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return set_error(PKV_EINVAL, "%s: num_tokens < 0", who);
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
    return set_error(PKV_EINVAL, "%s: null pointer", who);
  const int kv = desc->cache_dtype;
  if (kv == PKV_FP8_E4M3 || kv == PKV_INT8) {
    if (dtype_new != PKV_F32 && dtype_new != PKV_BF16)
      return set_error(PKV_EDTYPE, "%s: FP8/INT8 cache takes F32 or BF16 input", who);
    if (!k_scales || !v_scales)
      return set_error(PKV_EINVAL, "%s: FP8/INT8 cache needs scales", who);
  } else if (dtype_new != kv) {
    return set_error(PKV_EDTYPE, "%s: input dtype must equal the cache dtype", who);
  }
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return set_error(PKV_EALIGN, "%s: inputs and pools must be 16-byte aligned", who);
  AppendArgs a{};
  a.k_new = k_new;
  a.v_new = v_new;
  a.slots = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.num_tokens = num_tokens;
  a.h_kv = desc->num_kv_heads;
  a.head_dim = desc->head_dim;
  a.num_slots = (int64_t)desc->num_pages * desc->page_size;
  st = error_word(&a.err);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced("kv_append", s, [&] { return launch_kv_append(a, dtype_new, kv, s); });
  return cuda_status(e, "kv_append launch");
}

static int absmax_scales(const char* who, const void* x, int32_t dtype, int64_t n_tokens,
                         int32_t num_kv_heads, int32_t head_dim, float code_max,
                         float* scales_out, void* stream) {
  if (n_tokens < 0 || num_kv_heads <= 0 || (head_dim != 64 && head_dim != 128) || !scales_out ||
      (n_tokens > 0 && !x))
    return set_error(PKV_EINVAL, "%s: bad argument", who);
  if (dtype != PKV_F32 && dtype != PKV_BF16)
    return set_error(PKV_EDTYPE, "%s: x must be F32 or BF16", who);
  if (n_tokens > 0 && !aligned16(x)) return set_error(PKV_EALIGN, "%s: x alignment", who);
  if (reinterpret_cast<uintptr_t>(scales_out) & 3u)
    return set_error(PKV_EALIGN, "%s: scales_out alignment", who);
  if (num_kv_heads > 65535) return set_error(PKV_ESHAPE, "%s: too many heads", who);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced("kv_absmax", s, [&] {
    return launch_kv_absmax(x, dtype, n_tokens, num_kv_heads, head_dim, code_max, scales_out, s);
  });
  return cuda_status(e, "kv_absmax launch");
}

int pkv_kv_absmax_scales(const void* x, int32_t dtype, int64_t n_tokens, int32_t num_kv_heads,
                         int32_t head_dim, float* scales_out, void* stream) {
  return absmax_scales("pkv_kv_absmax_scales", x, dtype, n_tokens, num_kv_heads, head_dim, 448.f,
                       scales_out, stream);
}

int pkv_kv_absmax_scales_int8(const void* x, int32_t dtype, int64_t n_tokens,
                              int32_t num_kv_heads, int32_t head_dim, float* scales_out,
                              void* stream) {
  return absmax_scales("pkv_kv_absmax_scales_int8", x, dtype, n_tokens, num_kv_heads, head_dim,
                       127.f, scales_out, stream);
}

int pkv_copy_pages(void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                   const int32_t* src_pages, const int32_t* dst_pages, int32_t n, void* stream) {
  const char* who = "pkv_copy_pages";
  int st = check_desc(desc, who);
  if (st != PKV_OK) return st;
  if (n < 0) return set_error(PKV_EINVAL, "%s: n < 0", who);
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_pages || !dst_pages)
    return set_error(PKV_EINVAL, "%s: null pointer", who);
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return set_error(PKV_EALIGN, "%s: pools must be 16-byte aligned", who);
  const int eb = desc->cache_dtype == PKV_F32 ? 4 : desc->cache_dtype == PKV_BF16 ? 2 : 1;
  const int64_t page_bytes = (int64_t)desc->num_kv_heads * desc->page_size * desc->head_dim * eb;
  int* err = nullptr;
  st = error_word(&err);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced("copy_pages", s, [&] {
    return launch_copy_pages(k_cache, v_cache, src_pages, dst_pages, n, page_bytes,
                             desc->num_pages, err, s);
  });
  return cuda_status(e, "copy_pages launch");
}

int pkv_device_error(void* stream, int32_t* code_out) {
  if (!code_out) return set_error(PKV_EINVAL, "pkv_device_error: code_out is NULL");
  int* w = nullptr;
  int st = error_word(&w);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, w, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  st = cuda_status(e, "pkv_device_error");
  if (st != PKV_OK) return st;
  *code_out = v;
  if (v != 0) return set_error(PKV_EDEVICE, "device error word 0x%x", v);
  return PKV_OK;
}

int pkv_trace_enable(int on) {
  g_trace_on.store(on != 0);
  return PKV_OK;
}

int pkv_trace_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& r : g_trace) {
    cudaEventSynchronize(r.end);
    cudaEventDestroy(r.begin);
    cudaEventDestroy(r.end);
  }
  g_trace.clear();
  return PKV_OK;
}

int pkv_trace_read(const char* kernel, int32_t* launches_out, double* total_ms_out) {
  if (!kernel || !launches_out || !total_ms_out)
    return set_error(PKV_EINVAL, "pkv_trace_read: null pointer");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  int32_t n = 0;
  double total = 0.0;
  for (auto& r : g_trace) {
    if (r.name != kernel) continue;
    cudaError_t e = cudaEventSynchronize(r.end);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.begin, r.end);
    if (e != cudaSuccess) return cuda_status(e, "pkv_trace_read");
    ++n;
    total += ms;
  }
  *launches_out = n;
  *total_ms_out = total;
  return PKV_OK;
}

}  // extern "C"
