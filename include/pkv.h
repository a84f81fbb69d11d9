/*
 * pkv.h -- C ABI of the paged KV-cache library for sm_103a (GB300).
 *
 * What the library computes is the decode step of a KV-cached transformer layer over a
 * paged cache, as the KV-cache pages describe it:
 *  - "KV cache and PagedAttention", section 1 (The setup): at each generation step the new
 *    token's K and V are appended to the cache and attention of the new token's query reads
 *    the whole cached K and V. The "KV Cache" glossary calls these the write phase and the
 *    read phase.
 *  - Same page, section 4 (PagedAttention): the cache is a pool of fixed-size pages (16
 *    tokens); each request has a page table listing its page indices; the attention kernel
 *    gathers K/V through that table; the allocator is O(1); requests with a common prefix
 *    share pages.
 *  - "KV Cache" glossary, GQA and MQA paragraphs: a group of query heads shares one KV head.
 *  - Section 7 (KV cache quantisation): an FP8 (E4M3) cache at half the memory.
 *
 * Conventions for every entry point
 *  - Return value: PKV_OK (0) or a negative pkv_status. No exception or abort crosses the
 *    ABI. pkv_last_error() gives a message for the calling thread's last failure.
 *  - "device" pointers are CUDA device (or managed) memory of the current device, owned by
 *    the caller (kernels are launched on the current device); "host" pointers are ordinary
 *    host memory owned by the caller. A pointer is used only by the call that received it
 *    and by the GPU work that call enqueues (the TMA descriptors of a pool are cached by its
 *    address and shape; a new pool at the same address with the same shape reuses them
 *    correctly). The library never allocates device memory.
 *  - A call with nothing to do (a batch or token count of 0) returns PKV_OK at once and
 *    launches nothing; its buffer pointers may then be NULL (empty tensors have no storage).
 *  - stream is a cudaStream_t (NULL = the legacy default stream). GPU work is enqueued
 *    asynchronously on it; argument errors are detected on the host before anything is
 *    launched and nothing is launched then.
 *  - The GPU entry points may be called from several host threads at once (their launch
 *    caches and the split autotuner's records are locked). A call works on the device current
 *    in its thread and, if that thread has no CUDA context yet, makes the device's primary
 *    context current there (cudaSetDevice); a context already current is left as it is. The
 *    host-side objects (allocator, request tables, prefix cache) are not thread-safe.
 *  - Device-side faults of the data (a page id or slot outside the pool) never trap: the
 *    kernel skips the access and sets a bit in the device error word of the current device,
 *    which pkv_device_error() reads and clears.
 *
 * Pool layout (reading: the pages fix none): k_cache and v_cache are each
 *   [num_pages][num_kv_heads][page_size][head_dim]
 * elements of cache_dtype, so the 16 rows of one (page, KV head) form one contiguous tile.
 * Token position p of a request lives in page block_table[p / page_size], row
 * p % page_size; its slot is page * page_size + row.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,   /* bad argument value (null pointer, negative size, unsupported option) */
  PKV_ESHAPE = -2,   /* inconsistent sizes (head counts, head_dim, page size) */
  PKV_EDTYPE = -3,   /* unsupported dtype or dtype combination */
  PKV_EALIGN = -4,   /* a device pointer is not 16-byte aligned */
  PKV_ENOPAGES = -5, /* allocator: not enough free pages (nothing was allocated) */
  PKV_EREFCNT = -6,  /* allocator: page id out of range or reference count would underflow */
  PKV_ECUDA = -7,    /* a CUDA runtime call failed (message has the CUDA error string) */
  PKV_EDEVICE = -8,  /* the device error word was non-zero (see pkv_device_error) */
  PKV_ETIMEOUT = -9  /* reserved: a kernel wait timed out (reported in the error word) */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2, PKV_INT8 = 3 } pkv_dtype;

/* Bits of the device error word. */
enum {
  PKV_DEVERR_BAD_PAGE = 1, /* a block-table entry outside [0, num_pages), or a context longer
                              than its block-table row: the page is skipped */
  PKV_DEVERR_BAD_SLOT = 2, /* a slot outside [0, num_pages * page_size): token not written */
  PKV_DEVERR_TIMEOUT = 4,  /* a bounded wait on a shared-memory barrier gave up */
  PKV_DEVERR_BAD_GROUP = 8 /* cascade decode: inconsistent groups (a member whose context does
                              not extend past the shared prefix, a member index outside the
                              batch, more members or prefix pages than declared) */
};

/* Description of one layer's pair of pools. page_size must be 16; head_dim 64 or 128. */
typedef struct {
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t cache_dtype; /* pkv_dtype */
} pkv_cache_desc;

/* Message for the calling thread's last failed call ("" if none). Owned by the library. */
const char* pkv_last_error(void);

/* ABI version of this header: 1. */
int pkv_version(void);

/*
 * Write phase ("KV Cache" glossary: new K and V are appended to the cache; PagedAttention
 * section 4: they land in the request's page). For i < num_tokens and every KV head h:
 *   k_cache[slot / P][h][slot % P][:] = k_new[i][h][:]   (likewise v), slot = slot_mapping[i]
 * A negative slot skips token i (padding). A slot >= num_pages * P sets
 * PKV_DEVERR_BAD_SLOT and skips the token.
 *  k_new, v_new   device, [num_tokens][num_kv_heads][head_dim] of dtype_new, contiguous,
 *                 16-byte aligned.
 *  dtype_new      must equal cache_dtype for F32/BF16 caches; F32 or BF16 for an FP8/INT8
 *                 cache.
 *  slot_mapping   device int64 [num_tokens].
 *  k_cache,v_cache device pools (layout above), 16-byte aligned.
 *  k_scales, v_scales  device float [num_kv_heads], FP8/INT8 cache only (else ignored, may
 *                 be NULL). FP8: the stored code is round-to-nearest-even, saturating to
 *                 +-448, of the fp32 quotient x / scale[h] (section 7, "fp8 KV (E4M3)").
 *                 INT8 (section 7, "INT8 KV: similar"): the nearest integer (ties to even) of
 *                 the fp32 quotient, clamped to [-127, 127]. Rounding, saturation and the
 *                 symmetric INT8 range are this library's reading.
 */
int pkv_kv_append(const void* k_new, const void* v_new, int32_t dtype_new, int32_t num_tokens,
                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                  const pkv_cache_desc* desc, const float* k_scales, const float* v_scales,
                  void* stream);

/*
 * Bytes of device workspace pkv_paged_decode_attention needs for these sizes (0 when the
 * whole of every sequence is handled in one pass). max_pages_per_seq is the block-table
 * width. The result depends on the chunk size in force (pkv_decode_set_chunk_pages).
 */
size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_pages_per_seq);

/*
 * Read phase: single-token decode attention over the paged cache (section 1: only the new
 * token's query; attention over all cached K, V -- "cached + new", so context_lens counts
 * the token appended this step). For request b and query head h, with G = num_q_heads /
 * num_kv_heads and KV head j = h / G (consecutive groups; reading, the pages give none):
 *   s_t   = scale * <q[b][h], K_t>            for t < context_lens[b]
 *   out[b][h] = sum_t softmax(s)_t * V_t
 * where K_t, V_t are row t % P of page block_tables[b][t / P] (times k_scales[j] /
 * v_scales[j] for an FP8/INT8 cache). Accumulation is fp32. context_lens[b] == 0 gives out = 0.
 *  q            device [batch][num_q_heads][head_dim] of dtype_q (F32 or BF16).
 *               F32 q needs an F32, FP8 or INT8 cache; BF16 q a BF16, FP8 or INT8 cache.
 *  block_tables device int32 [batch][max_pages_per_seq]; entries past a request's last page
 *               are not read.
 *  context_lens device int32 [batch], each <= max_pages_per_seq * 16 (longer ones are cut
 *               to that and flagged with PKV_DEVERR_BAD_PAGE).
 *  out          device [batch][num_q_heads][head_dim] of dtype_q.
 *  workspace    device, >= pkv_decode_workspace_size(...) bytes, 16-byte aligned, or NULL
 *               when that size is 0. It must be zero-filled before its first use; every call
 *               that completes leaves it zero-filled where that matters (reuse it freely on
 *               one stream; re-zero it after a call that reported a device error; one workspace
 *               per stream). Long contexts are split into chunks of pages whose partial results
 *               (running max, sum, weighted values) are merged in a fixed order -- by a
 *               second kernel, or by the last CTA of each group when chosen with
 *               pkv_decode_set_merge_in_place -- so results do not depend on physical page
 *               placement.
 * Requires num_q_heads % num_kv_heads == 0 and G in {1, 2, 4, 8, 16}.
 */
int pkv_paged_decode_attention(const void* q, int32_t dtype_q, int32_t batch,
                               int32_t num_q_heads, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* desc, const int32_t* block_tables,
                               int32_t max_pages_per_seq, const int32_t* context_lens,
                               float scale, const float* k_scales, const float* v_scales,
                               void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step, append and attention fused in one launch (write phase + read phase of
 * "KV cache and PagedAttention" section 1): for every request b with context_lens[b] >= 1,
 * the row k_new[b] / v_new[b] is written at position context_lens[b] - 1 (page
 * block_tables[b][p / 16], row p % 16), then attention runs over positions
 * 0 .. context_lens[b] - 1 exactly as pkv_paged_decode_attention. The pool bytes and the
 * output equal those of pkv_kv_append (with that position's slot) followed by
 * pkv_paged_decode_attention.
 *  k_new, v_new  device [batch][num_kv_heads][head_dim] of dtype_new, 16-byte aligned;
 *                dtype_new as for pkv_kv_append.
 * The page holding the new position must belong to request b alone (not a shared prefix page).
 * Other arguments as pkv_paged_decode_attention.
 */
int pkv_paged_decode_step(const void* q, int32_t dtype_q, int32_t batch, int32_t num_q_heads,
                          const void* k_new, const void* v_new, int32_t dtype_new,
                          void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                          const int32_t* block_tables, int32_t max_pages_per_seq,
                          const int32_t* context_lens, float scale, const float* k_scales,
                          const float* v_scales, void* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Sliding-window decode with attention sinks ("KV cache and PagedAttention", section 8: keep
 * only the last W tokens; attention sinks also keep the first few). With window > 0 a request
 * of ctx = context_lens[b] tokens attends positions t >= ctx - window and t < sink_tokens only;
 * pages holding no attended position are never read, so the caller may release them (their
 * block-table entries are then ignored). window == 0 is full attention (sink_tokens must then
 * be 0). Otherwise as pkv_paged_decode_attention / pkv_paged_decode_step.
 */
int pkv_paged_decode_attention_window(const void* q, int32_t dtype_q, int32_t batch,
                                      int32_t num_q_heads, const void* k_cache,
                                      const void* v_cache, const pkv_cache_desc* desc,
                                      const int32_t* block_tables, int32_t max_pages_per_seq,
                                      const int32_t* context_lens, float scale,
                                      const float* k_scales, const float* v_scales,
                                      int32_t sink_tokens, int32_t window, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);
int pkv_paged_decode_step_window(const void* q, int32_t dtype_q, int32_t batch,
                                 int32_t num_q_heads, const void* k_new, const void* v_new,
                                 int32_t dtype_new, void* k_cache, void* v_cache,
                                 const pkv_cache_desc* desc, const int32_t* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* context_lens,
                                 float scale, const float* k_scales, const float* v_scales,
                                 int32_t sink_tokens, int32_t window, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * The same decode attention as pkv_paged_decode_attention, for callers that cannot allocate
 * device memory (a plugin whose host application owns all device memory and gives it no
 * allocation hook; a server that reserved all free HBM for its KV pools at start-up; a
 * latency-critical loop that must not risk cudaMalloc's device-wide synchronisation). It takes
 * no workspace: the split partials go to a 16 MiB scratch array built into the library, held in
 * device memory on every GPU that loads the library until the process exits. The pages have no
 * counterpart to this entry point; it is a deployment convenience of this library.
 *  - Arguments, layouts and results are those of pkv_paged_decode_attention.
 *  - Sizes whose split would need more than the scratch (pkv_decode_workspace_size(...) >
 *    pkv_decode_noalloc_scratch_bytes()) are rejected with PKV_EINVAL before anything runs.
 *  - Calls no cudaMalloc or cudaFree. The first call on a device looks up the scratch's device
 *    address for that device (with it current); make that call before any stream capture.
 *    The address is kept per device and context: after a cudaDeviceReset the next call looks
 *    it up again.
 *  - All calls on a device share the scratch and it keeps the last call's contents; each call
 *    zeroes the small part that must start at zero. Calls whose kernels may overlap on the GPU,
 *    e.g. on two streams without ordering between them, race on it; calls on one stream are
 *    safe.
 */
int pkv_paged_decode_attention_noalloc(const void* q, int32_t dtype_q, int32_t batch,
                                       int32_t num_q_heads, const void* k_cache,
                                       const void* v_cache, const pkv_cache_desc* desc,
                                       const int32_t* block_tables, int32_t max_pages_per_seq,
                                       const int32_t* context_lens, float scale,
                                       const float* k_scales, const float* v_scales, void* out,
                                       void* stream);

/* Bytes of the scratch pkv_paged_decode_attention_noalloc uses (16 MiB). */
size_t pkv_decode_noalloc_scratch_bytes(void);

/*
 * Copy whole pages of both pools (every KV head): for p < n, page dst_pages[p] becomes a copy
 * of page src_pages[p] (device int32 arrays). With pkv_cow_page this gives copy-on-write for
 * pages shared across sequences ("KV Cache" glossary: blocks shared for parallel sampling and
 * beam search; the copy rule is this library's reading). An id outside [0, num_pages) skips
 * that page and sets PKV_DEVERR_BAD_PAGE. Source and destination pages must not overlap.
 */
int pkv_copy_pages(void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                   const int32_t* src_pages, const int32_t* dst_pages, int32_t n, void* stream);

/*
 * Per-KV-head scales for an FP8 cache (section 7; granularity is this library's reading):
 *   scales_out[h] = fp32(max |x[:, h, :]| / 448), or 1 if that maximum is 0.
 *  x           device [n_tokens][num_kv_heads][head_dim] of dtype (F32 or BF16), 16-byte
 *              aligned.
 *  scales_out  device float [num_kv_heads]; overwritten.
 */
int pkv_kv_absmax_scales(const void* x, int32_t dtype, int64_t n_tokens, int32_t num_kv_heads,
                         int32_t head_dim, float* scales_out, void* stream);
/* The same for an INT8 cache: scales_out[h] = fp32(max |x[:, h, :]| / 127), or 1. */
int pkv_kv_absmax_scales_int8(const void* x, int32_t dtype, int64_t n_tokens,
                              int32_t num_kv_heads, int32_t head_dim, float* scales_out,
                              void* stream);

/*
 * Synchronises stream, then reads and clears the current device's error word into
 * *code_out (host). Returns PKV_OK, or PKV_EDEVICE when the word was non-zero. The word is
 * shared by every stream of the device in this process.
 */
int pkv_device_error(void* stream, int32_t* code_out);

/* Largest chunk of the split over pages, in pages (1..4096); each sequence is cut into the
 * fewest near-equal chunks no larger than this. 0 restores the automatic choice.
 * Process-wide; affects calls made after it returns. */
int pkv_decode_set_chunk_pages(int32_t pages);

/* Merge the chunks of a split sequence inside the decode kernel (the last CTA of each
 * (request, KV head) to finish merges them, using a counter in the workspace) when the call has
 * at most max_chunks chunks per sequence; 0 (the default) always uses the separate combine
 * kernel, which measured faster on every workload tried. Process-wide. */
int pkv_decode_set_merge_in_place(int32_t max_chunks);

/* Which decode kernel pkv_paged_decode_attention uses: 0 = automatic (tensor cores for a bf16,
 * FP8 or INT8 cache with head_dim 128, CUDA cores otherwise), 1 = always the CUDA-core kernel,
 * 2 = always the tensor-core kernel (calls it cannot serve then fail with PKV_EINVAL).
 * Process-wide; affects calls made after it returns. Both kernels compute the same result
 * within the documented tolerances; each is deterministic for a given choice. */
int pkv_decode_set_kernel(int32_t which);

/* How the tensor-core decode splits a call that needs split partials (workspace size > 0).
 * The splits, each merged by a combine kernel in a fixed order:
 *  - chunks, as described under pkv_paged_decode_attention (a CTA per (request, KV head,
 *    chunk); the hardware hands out CTAs as SMs free up);
 *  - chunks 1.5 or 2 times the automatic length (fewer CTAs and waves of them; the partials
 *    fit the same slots), when the chunk size is automatic;
 *  - balanced: the whole call's (request, KV head, attended page) stream is cut into equal
 *    contiguous shares, one per warp of a single wave of CTAs (no more warps than the workspace
 *    has partial slots for), and each (request, KV head)'s partials are merged in stream order.
 *    It applies when the chunk size is automatic (pkv_decode_set_chunk_pages(0)), partials go
 *    to the combine kernel, batch <= 2048 and the call is not a cascade decode. Under it a
 *    request's split (and so its rounding) depends on the whole batch's lengths, not on
 *    physical page placement.
 * mode 0 = automatic (the default): the split recorded for the call's shape by autotuning
 * (pkv_decode_set_autotune), else chunks; 1 = chunks only; 2 = balanced wherever it applies;
 * 3, 4 = chunks 1.5 or 2 times longer wherever they apply.
 * Results are deterministic for given inputs and choice. Process-wide. */
int pkv_decode_set_split(int32_t mode);

/* Autotuning of the split (mode 0): while on, the first call of each shape -- cache and query
 * dtypes, batch, head counts, table width, window and sinks, fused append or not -- for which
 * more than one split applies runs the decode five times with each split that applies, in
 * turn, on its stream, synchronises the stream, records the split whose decode kernel took the
 * least time (the combine is not timed) and gives its result. Later calls of that shape use the
 * recorded split without timing. Calls made while their stream is being captured into a CUDA
 * graph never time (they use the recorded split, else chunks); so do calls on a device other
 * than the one current when autotuning was turned on (its timing events are made then, so
 * decode calls create nothing). Off by default. */
int pkv_decode_set_autotune(int32_t on);

/* Forgets every recorded split. */
int pkv_decode_autotune_reset(void);

/* The split recorded for a shape: 0 chunks, 1 balanced, 2 and 3 chunks 1.5 and 2 times
 * longer, -1 none recorded. */
int pkv_decode_split_choice(int32_t kv_dtype, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t max_pages_per_seq, int32_t window,
                            int32_t sink_tokens, int32_t fused);

/* Largest chunk (pages) the decode uses for these sizes under the current setting. */
int32_t pkv_decode_chunk_pages(int32_t batch, int32_t num_kv_heads, int32_t max_pages_per_seq);

/* ---- host page accounting (no GPU needed) ------------------------------------------------ */

/* Pages a request of n_tokens occupies: the smallest count whose capacity holds it (section 4:
 * a 17-token request uses 2 pages of 16). */
int pkv_pages_needed(int64_t n_tokens, int32_t page_size, int64_t* pages_out);

/*
 * Slots of n tokens: token i is position positions[i] of request requests[i] (requests may be
 * NULL, meaning request i). slots_out[i] = block_tables[r][p / P] * P + p % P, or -1 when
 * p < 0. All host arrays. Fails with PKV_EINVAL (slots_out unspecified) when p / P >=
 * max_pages_per_seq or the table entry is outside [0, num_pages).
 */
int pkv_slot_mapping(const int32_t* block_tables, int32_t max_pages_per_seq,
                     const int32_t* requests, const int64_t* positions, int64_t n,
                     int32_t page_size, int32_t num_pages, int64_t* slots_out);

/*
 * Page allocator (section 4: uniform pages, O(1) allocator; shared pages for prefixes).
 * A LIFO free list plus one reference count per page; every operation is O(1) per page and
 * all-or-nothing. Not thread-safe: one handle per thread or external locking.
 */
typedef struct pkv_allocator pkv_allocator;

/* initial_free_order (host, may be NULL = 0..num_pages-1) lists the pages in the order the
 * first allocations hand them out. */
int pkv_allocator_create(int32_t num_pages, const int32_t* initial_free_order,
                         pkv_allocator** out);
/* Frees the allocator's own bookkeeping (the pools are the caller's device memory). Objects
 * built on it (request tables, prefix caches) must be destroyed first. */
void pkv_allocator_destroy(pkv_allocator* a);
/* n pages with reference count 1 into page_ids_out (host); PKV_ENOPAGES if fewer are free. */
int pkv_alloc(pkv_allocator* a, int32_t n, int32_t* page_ids_out);
/* One more reference to each listed (allocated) page: sharing a prefix. */
int pkv_incref(pkv_allocator* a, const int32_t* ids, int32_t n);
/* One reference less to each listed page; a page reaching 0 returns to the free list.
 * PKV_EREFCNT (nothing changed) if an id is out of range or would drop below 0. */
int pkv_decref(pkv_allocator* a, const int32_t* ids, int32_t n);
/* Copy-on-write before writing position `position` of a request whose pages are row[0..n)
 * (host array): if the page holding it is shared (reference count > 1) it is replaced in row by
 * a newly allocated page, the old page loses this request's reference, and *copy_src and *copy_dst
 * name the page contents to copy (pkv_copy_pages) before the write; otherwise both are -1
 * (also when the position starts a page the request does not have yet). */
int pkv_cow_page(pkv_allocator* a, int32_t* row, int32_t n, int64_t position, int32_t page_size,
                 int32_t* copy_src, int32_t* copy_dst);
/* Number of free pages (-1 for NULL). */
int32_t pkv_num_free(const pkv_allocator* a);
/* Reference count of a page, or -1 for an id out of range. */
int32_t pkv_refcount(const pkv_allocator* a, int32_t id);

/*
 * Request page tables over an allocator (section 4: a page table per request; section 5:
 * requests join and leave every step; section 6 and the "KV Cache" glossary: prefixes, parallel
 * samples and beams share pages; section 8: pages outside a sliding window are released).
 * A request (any int64 id) is a row of page ids (-1 where a page was released) and a token
 * count; every page in a row holds one allocator reference. Host only; not thread-safe. The
 * table does not own the allocator, which must outlive it; destroying the table drops its
 * rows without touching the allocator (free the requests first to return their pages).
 * Calls that fail with PKV_EINVAL or PKV_ENOPAGES change nothing.
 */
typedef struct pkv_seq_table pkv_seq_table;
int pkv_seq_table_create(pkv_allocator* a, int32_t page_size, pkv_seq_table** out);
void pkv_seq_table_destroy(pkv_seq_table* t);
/* A new request, empty or starting on n_shared whole pages holding its first shared_len =
 * n_shared * page_size tokens (a cached prefix; one more reference on each). */
int pkv_seq_add(pkv_seq_table* t, int64_t rid, const int32_t* shared_pages, int32_t n_shared,
                int64_t shared_len);
/* The same, but the request takes over references the caller already holds on the pages
 * (for example those a prefix-cache lookup handed out) instead of taking new ones. */
int pkv_seq_adopt(pkv_seq_table* t, int64_t rid, const int32_t* pages, int32_t n_pages,
                  int64_t n_tokens);
/* new_rids[i] becomes a copy of src_rids[i] (same pages, one more reference on each, same
 * length), in order: a parent may be a request forked earlier in the list. */
int pkv_seq_fork(pkv_seq_table* t, const int64_t* src_rids, const int64_t* new_rids, int32_t n);
/* Drops the listed requests and their page references. */
int pkv_seq_free(pkv_seq_table* t, const int64_t* rids, int32_t n);
/*
 * Grows request rids[i] by counts[i] tokens, in order. For a request with counts[i] > 0 whose
 * next position falls in a shared page, the page is first replaced by a fresh one
 * (pkv_cow_page) and the pair (old, new) is appended to copy_src/copy_dst (host, room for n
 * pairs; the caller copies the contents on the device, pkv_copy_pages, before the writes);
 * *n_copies receives their number. Then the pages the new length needs are allocated. The
 * slots of the new positions, request by request, go to slots_out (host, sum of counts):
 * page * page_size + position % page_size. PKV_ENOPAGES (nothing changed) when the free pages
 * cannot cover every copy and page of the batch; PKV_EINVAL for an unknown or repeated id, a
 * negative count or a write into a released page.
 */
int pkv_seq_reserve(pkv_seq_table* t, const int64_t* rids, const int32_t* counts, int32_t n,
                    int64_t* slots_out, int32_t* copy_src, int32_t* copy_dst, int32_t* n_copies);
/* Block-table rows (int32 [n][width], unused columns 0) and token counts (int32 [n]) of the
 * listed requests into host arrays (either may be NULL). PKV_EINVAL if a row does not fit. */
int pkv_seq_tables(const pkv_seq_table* t, const int64_t* rids, int32_t n, int32_t width,
                   int32_t* block_tables_out, int32_t* context_lens_out);
/*
 * One scheduler step in one call ("KV cache and PagedAttention", section 5: requests leave and
 * join the running batch every step). In order: the n_free finished requests are dropped
 * (pkv_seq_free); the n_new new requests are added empty and grown by their prompt_counts
 * tokens (their slots, request by request, to prompt_slots_out: host, sum of prompt_counts);
 * every one of the n_live live requests -- which may include new ones -- is grown by one token
 * (slots to live_slots_out, host [n_live], or NULL), with copy-on-write as in pkv_seq_reserve
 * (copy_src/copy_dst: host, room for n_live pairs, or NULL when no live page is shared
 * once the frees are done -- references held by the finished requests do not count;
 * *n_copies set); and their block-table rows and token counts are written as by
 * pkv_seq_tables (block_tables_out [n_live][width] and context_lens_out [n_live], host,
 * either may be NULL). With incremental != 0, a row that already holds the same request's
 * row from the previous incremental step into the same buffer with the same width is
 * written only from the first column that changed since (new pages, copies, released
 * pages); every other row in full. The caller then must not change those rows in between
 * (a pkv_seq_tables call into the same buffer pointer makes the next step write in full).
 * Every argument is checked before anything changes (PKV_EINVAL: an
 * unknown or repeated id, a new id that is live, a live id that is neither live nor new, a
 * write into a released page, a row wider than the table). The frees then stand; if the pages
 * cannot cover the prompts, the copies and the new tokens (PKV_ENOPAGES), the new requests
 * are removed again and their pages returned (the free list's order may differ), so the
 * table holds exactly the state after the frees. Not thread-safe.
 */
int pkv_seq_step(pkv_seq_table* t, const int64_t* free_rids, int32_t n_free,
                 const int64_t* new_rids, const int32_t* prompt_counts, int32_t n_new,
                 int64_t* prompt_slots_out, const int64_t* live_rids, int32_t n_live,
                 int64_t* live_slots_out, int32_t width, int32_t* block_tables_out,
                 int32_t* context_lens_out, int32_t incremental, int32_t* copy_src,
                 int32_t* copy_dst, int32_t* n_copies);
/* The table width (columns) a pkv_seq_step with these new requests, prompts and live requests
 * needs: the most pages any live request holds after it grows by its prompt (a new request)
 * and one token -- ceil((length + 1) / page_size), or more where it already holds more rows --
 * and at least 1. Host arrays; PKV_EINVAL for an unknown live id that is not new, or a
 * negative prompt. Changes nothing. */
int pkv_seq_step_width(const pkv_seq_table* t, const int64_t* new_rids,
                       const int32_t* prompt_counts, int32_t n_new, const int64_t* live_rids,
                       int32_t n_live, int32_t* width_out);
/* Releases every page of the request whose positions all lie at or past sink_tokens, before
 * the last `window` positions and before the newest token (window 0: none); their row entries
 * become -1. *released (may be NULL) receives the count. */
int pkv_seq_release_outside_window(pkv_seq_table* t, int64_t rid, int64_t window,
                                   int64_t sink_tokens, int32_t* released);
/* Token count of a request, or -1 if unknown. */
int64_t pkv_seq_len(const pkv_seq_table* t, int64_t rid);
/* Row length of a request (or -1 if unknown); copies up to cap entries into pages_out. */
int32_t pkv_seq_pages(const pkv_seq_table* t, int64_t rid, int32_t* pages_out, int32_t cap);
/* Number of requests; pkv_seq_ids copies up to cap ids (any order) and returns the number. */
int32_t pkv_seq_count(const pkv_seq_table* t);
int32_t pkv_seq_ids(const pkv_seq_table* t, int64_t* rids_out, int32_t cap);

/* ---- decode step from host memory ---------------------------------------------------------- */

/*
 * Layout of the packed step inputs (host): q [batch][num_q_heads][head_dim] (dtype_q), k_new and
 * v_new [batch][num_kv_heads][head_dim] (dtype_new), block_tables int32 [batch][max_pages],
 * context_lens int32 [batch], each starting at offsets[0..4] (256-byte aligned, in this order);
 * *total_bytes is the size of the block.
 */
int pkv_packed_step_layout(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t max_pages_per_seq, int32_t dtype_q,
                           int32_t dtype_new, size_t* offsets, size_t* total_bytes);

/*
 * pkv_paged_decode_step_window with its inputs and output in host memory (window = 0, sinks 0:
 * pkv_paged_decode_step): one copy of the packed inputs (host_in, pinned, laid out as
 * pkv_packed_step_layout says) into dev_in (device, the same size), the fused append + decode
 * on the device copies, and one copy of the output (out_dev, device) into out_host (pinned
 * for an asynchronous copy; any host memory works), all on `stream` (the caller synchronises
 * before reading out_host or rewriting host_in).
 */
int pkv_paged_decode_step_packed(const void* host_in, void* dev_in, int32_t batch,
                                 int32_t num_q_heads, int32_t dtype_q, int32_t dtype_new,
                                 void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                 int32_t max_pages_per_seq, float scale, const float* k_scales,
                                 const float* v_scales, int32_t sink_tokens, int32_t window,
                                 void* out_dev, void* out_host, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ---- cascade decode (shared prompt prefixes) ---------------------------------------------- */

/*
 * Requests whose page tables start with the same physical pages (a shared prompt prefix,
 * "KV cache and PagedAttention" section 6; "KV Cache" glossary, prefix caching) form groups.
 * The cascade decode computes the attention of every member's query heads over the group's
 * shared pages once per group -- the pages are read once for all members, and the members'
 * queries form a dense tensor-core contraction -- then over each member's own pages, and
 * merges the two with the split-decode rule (a softmax over a union of disjoint key sets from
 * the per-set maxima, sums and weighted values): in the combine kernel, or in the own-page
 * kernel (see pkv_cascade_set_overlap). The result is the same attention as
 * pkv_paged_decode_attention over the same tables (rounding aside).
 *
 * Arrays are device memory unless noted; the bounds are host values that the arrays must
 * respect (the kernels clamp to them and flag PKV_DEVERR_BAD_GROUP otherwise).
 */
typedef struct {
  const int32_t* group_of;       /* [batch]: group of request b, or -1 */
  const int32_t* prefix_pages;   /* [n_groups]: leading pages shared by every member of g */
  const int32_t* group_offsets;  /* [n_groups + 1]: members of g are ... */
  const int32_t* group_members;  /* ... group_members[group_offsets[g] .. group_offsets[g+1]) */
  int32_t n_groups;              /* 0: a plain decode */
  int32_t max_members;           /* host: most members of any group, in [1, batch] */
  int32_t max_prefix_pages;      /* host: most shared pages of any group, in [1, table width] */
  int32_t max_own_pages;         /* host hint: most pages any request reads past its group's
                                    shared pages (all its pages outside a group); sizes the
                                    split of those pages. 0: the table width. A request with
                                    more pages still gets a correct result, in larger chunks. */
  const int32_t* own_start;      /* [batch] or NULL: prefix_pages[group_of[b]] (0 outside a
                                    group), read directly by the decode of the members' own
                                    pages instead of through group_of (one read fewer) */
  const int32_t* prefix_page_ids; /* [n_groups][max_prefix_pages] or NULL: group g's shared
                                    page ids (its members' first table entries), so that the
                                    prefix pass reads them directly instead of through
                                    group_members and the first member's table row
                                    (pkv_cascade_prefix_page_ids fills it) */
} pkv_cascade_desc;

/*
 * Host. Groups of a batch from its HOST page tables [batch][max_pages_per_seq] and context
 * lengths: requests are bucketed by their first page id (batch order); a bucket of at least
 * min_members (>= 2) requests shares the longest run of leading page ids common to all its
 * members, cut to the full pages before each member's position ctx - 1; fewer than
 * min_prefix_pages (>= 1) shared pages: no group. Outputs (host, caller-sized): group_of
 * [batch], prefix_pages [batch], group_offsets [batch + 1], group_members [batch], own_start
 * [batch] (may be NULL), and the
 * counts and bounds of a pkv_cascade_desc (*n_groups may be 0; *max_own_pages counts the pages
 * of a context cut to the table width). Its working arrays are kept per host thread between
 * calls (a call allocates nothing once a batch of that size has been seen); calls from
 * different threads do not share them.
 */
int pkv_cascade_groups(const int32_t* block_tables, const int32_t* context_lens, int32_t batch,
                       int32_t max_pages_per_seq, int32_t min_members, int32_t min_prefix_pages,
                       int32_t* group_of, int32_t* prefix_pages, int32_t* group_offsets,
                       int32_t* group_members, int32_t* n_groups, int32_t* max_members,
                       int32_t* max_prefix_pages, int32_t* max_own_pages, int32_t* own_start);

/* The shared page ids of each group, [n_groups][max_prefix_pages] (row g: the first
 * prefix_pages[g] entries of its first member's table row, the rest -1), from the host arrays
 * pkv_cascade_groups wrote for block_tables [batch][max_pages_per_seq]; ids_out is host memory
 * of n_groups * max_prefix_pages int32. PKV_EINVAL for a group without members, a member
 * outside [0, batch) or more shared pages than max_prefix_pages. */
int pkv_cascade_prefix_page_ids(const int32_t* block_tables, int32_t batch,
                                int32_t max_pages_per_seq, const int32_t* prefix_pages,
                                const int32_t* group_offsets, const int32_t* group_members,
                                int32_t n_groups, int32_t max_prefix_pages, int32_t* ids_out);

/* Workspace bytes of a cascade decode (its partials: the prefix chunks, then the members' own
 * chunks, for every request); pkv_decode_workspace_size when groups has no group. Zero-fill it
 * before first use. */
size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_pages_per_seq,
                                  const pkv_cascade_desc* groups);

/* Pages per CTA of the prefix pass for these groups (0 without groups). */
int32_t pkv_cascade_prefix_chunk_pages(int32_t num_kv_heads, int32_t num_q_heads,
                                       const pkv_cascade_desc* groups);

/*
 * Cascade decode attention: the arguments of pkv_paged_decode_attention (bf16 cache and
 * queries, head_dim 128; no window) plus the groups. Every member's table must list its
 * group's shared pages first and its context must cover them. Launches the prefix kernel,
 * then the decode kernel over the members' own pages (and the other requests' pages), which
 * merges.
 * groups == NULL or n_groups == 0: exactly pkv_paged_decode_attention.
 */
int pkv_cascade_decode_attention(const void* q, int32_t dtype_q, int32_t batch,
                                 int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                 const pkv_cache_desc* desc, const int32_t* block_tables,
                                 int32_t max_pages_per_seq, const int32_t* context_lens,
                                 float scale, const pkv_cascade_desc* groups, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Cascade decode step: as pkv_paged_decode_step (the append of this step's K/V rows is fused
 * into the decode), with the groups; each member's context must extend past its shared pages. */
int pkv_cascade_decode_step(const void* q, int32_t dtype_q, int32_t batch, int32_t num_q_heads,
                            const void* k_new, const void* v_new, int32_t dtype_new,
                            void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                            const int32_t* block_tables, int32_t max_pages_per_seq,
                            const int32_t* context_lens, float scale,
                            const pkv_cascade_desc* groups, void* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * The cascade decode step from host memory. Layout of the block (host_in, pinned, and its
 * device twin dev_in, the same size): the five regions of pkv_packed_step_layout (offsets[0..4])
 * filled by the caller, then six int32 regions this call fills (offsets[5..10]): group_of
 * [batch], prefix_pages [batch], group_offsets [batch + 1], group_members [batch], own_start
 * [batch] and, last, the groups' shared page ids [batch / 2][max_pages_per_seq] (at most
 * batch / 2 groups), each 256-byte aligned; *total_bytes is the size of the block. A step
 * copies the block up to the end of the page ids its groups use.
 */
int pkv_packed_cascade_layout(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_pages_per_seq, int32_t dtype_q,
                              int32_t dtype_new, size_t* offsets, size_t* total_bytes);

/*
 * One call per step: groups the batch on the host from the block's page tables and context
 * lengths (pkv_cascade_groups, at least 2 members and 1 shared page per group) into the block's
 * group regions, copies the whole block into dev_in, runs pkv_cascade_decode_step on the device
 * copies (a plain fused decode step when no group forms) and copies the output (out_dev) into
 * out_host, all on `stream`. host_in is written (the group regions), so the caller
 * synchronises before rewriting it or reading out_host. The workspace must hold
 * pkv_cascade_workspace_size for this step's groups: *workspace_needed (may be NULL) receives
 * it, and a smaller workspace fails with PKV_EINVAL before anything is enqueued;
 * *n_groups_out (may be NULL) receives the number of groups.
 */
int pkv_cascade_decode_step_packed(void* host_in, void* dev_in, int32_t batch,
                                   int32_t num_q_heads, int32_t dtype_q, int32_t dtype_new,
                                   void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                   int32_t max_pages_per_seq, float scale, void* out_dev,
                                   void* out_host, void* workspace, size_t workspace_bytes,
                                   size_t* workspace_needed, int32_t* n_groups_out,
                                   void* stream);

/* Tuning: when every request of a tensor-core decode fits one chunk of at most 16 pages,
 * one warp serves each request (1, the default) or four warps share one (0). */
int pkv_decode_set_warp_per_request(int32_t on);

/* Tuning: in a cascade decode on the tensor-core path, the own-page decode is launched as a
 * programmatic dependent of the prefix kernel. 2 (the default): it writes each member's result
 * as a partial and exits without waiting (one thread of its first CTA waits for the prefix
 * kernel before exiting), the combine kernel merges prefix and own partials, and the tcgen05
 * prefix kernel is sized for about half the SMs so that the two kernels share the GPU. 1: it
 * waits for the prefix kernel before folding the prefix partials in itself (no combine).
 * 0 runs the two kernels one after the other. The results agree within rounding (mode 2
 * merges in another order). Process-wide; the workspace size depends on it. */
int pkv_cascade_set_overlap(int32_t on);

/* Tuning: pages per CTA of the prefix pass (0 = automatic). */
int pkv_cascade_set_prefix_chunk_pages(int32_t pages);

/* Tuning: the prefix pass on tcgen05 (tensor memory accumulators, 128 rows per CTA; 0 =
 * automatic, 2) or on mma.sync (64 rows per CTA; 1). Same results up to rounding. */
int pkv_cascade_set_prefix_kernel(int32_t which);

/* ---- prefix cache (host) ----------------------------------------------------------------- */

/*
 * Reuse of the KV pages of a prompt prefix ("KV cache and PagedAttention", section 6: hash the
 * prefix tokens, store its pages keyed by the hash, reuse them on a match; "KV Cache" glossary:
 * longest common prefix; pitfall 5: include the tenant in the key). Whole pages only: entry i
 * of a prompt is keyed by a chained hash of (tenant, tokens of pages 0..i) and stores its
 * tokens, so a match is exact (collisions never share pages). The cache holds one reference on
 * each listed page (through the allocator it was created with). Not thread-safe.
 */
typedef struct pkv_prefix_cache pkv_prefix_cache;
int pkv_prefix_cache_create(pkv_allocator* a, int32_t page_size, pkv_prefix_cache** out);
/* Drops the cache's page references. */
void pkv_prefix_cache_destroy(pkv_prefix_cache* c);
/* Longest cached prefix of tokens[0..n) in whole pages, at most max_pages: its page ids go to
 * pages_out (host) and *n_pages_out; the caller receives one reference on each. */
int pkv_prefix_lookup(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens, int64_t n,
                      int32_t* pages_out, int32_t max_pages, int32_t* n_pages_out);
/* Registers the full pages of a prompt: pages[i] holds tokens [i*P, (i+1)*P). Pages already
 * cached for the same prefix are kept (the caller's copies are not taken). */
int pkv_prefix_insert(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens, int64_t n,
                      const int32_t* pages, int32_t n_pages);
/* pkv_prefix_insert of request rid's own pages (a request table over the same allocator): the
 * full pages among the first min(n, its length) tokens, tokens[0..n) being its prompt. */
int pkv_prefix_insert_request(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens,
                              int64_t n, const pkv_seq_table* t, int64_t rid);
/* A new request rid in table t whose prompt is tokens[0..n): it starts on the pages of the
 * longest prefix the cache holds for this tenant (a pkv_prefix_lookup whose references the
 * request adopts, pkv_seq_adopt); *cached_tokens receives the prompt tokens already cached
 * (whole pages). On an error nothing changes and no reference is kept. */
int pkv_seq_add_cached_prefix(pkv_seq_table* t, int64_t rid, pkv_prefix_cache* c, int64_t tenant,
                              const int32_t* tokens, int64_t n, int64_t* cached_tokens);
/* Releases up to max_pages least recently used entries that end a cached chain and whose page
 * only the cache references; *n_evicted receives the count. */
int pkv_prefix_evict(pkv_prefix_cache* c, int32_t max_pages, int32_t* n_evicted);
/* Number of cached pages (-1 for NULL). */
int32_t pkv_prefix_size(const pkv_prefix_cache* c);

/* ---- tracing --------------------------------------------------------------------------------- */

/* When on, every kernel the library launches, and each copy of the packed host steps, is
 * bracketed by a pair of CUDA events on its stream. pkv_trace_read() synchronises those events
 * and reports, for the family named ("paged_decode", "decode_combine", "cascade_prefix",
 * "kv_append", "kv_absmax", "copy_pages", and the packed steps' "h2d_copy" and "d2h_copy"),
 * the number of launches and their summed device time in milliseconds since the last reset.
 * pkv_trace_reset() drops all records. */
int pkv_trace_enable(int on);
int pkv_trace_reset(void);
int pkv_trace_read(const char* kernel, int32_t* launches_out, double* total_ms_out);

/*
 * Self-test of the kernels' failure detection: one thread waits, with the same bounded wait
 * every kernel uses on its copy barriers, on a barrier that nothing completes. After the wait's
 * limit (2 s) it gives up: PKV_DEVERR_TIMEOUT is OR-ed into *err_dev and *done_dev is set to 1
 * (2 would mean the wait completed). err_dev and done_dev are device int32 words owned by the
 * caller; asynchronous on the stream. Nothing faults or hangs; the context stays usable.
 */
int pkv_selftest_wait_timeout(int32_t* err_dev, int32_t* done_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
