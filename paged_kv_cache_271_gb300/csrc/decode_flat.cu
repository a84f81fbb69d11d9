// Balanced split of the tensor-core decode ("KV cache and PagedAttention", sections 1 and 4:
// the read phase over every request's pages).
//
// The chunked decode gives every (request, KV head, chunk) its own CTA. Its CTAs are of equal
// size, so they start and finish in waves: every wave change leaves each SM's bandwidth half
// used while the new CTAs wait on their first context length, table row and page, and the
// last wave drains unevenly. Here the work is laid out as one stream instead -- every
// (request b, KV head j, attended page p) in order b, j, p -- and cut into equal contiguous
// shares, one per warp of a single wave of CTAs. A warp walks its share through its own
// ring stages without a break: the page ids and copies of the next request run ahead across
// the boundary. Each run of pages of one (b, j) -- a segment -- ends in
//  * the output itself, when the segment is the whole of (b, j);
//  * otherwise a partial (running max, sum, weighted values per head), which the combine
//    kernel merges in stream order.
// With T pages in the stream and N warps, warp w takes pages [w T / N, (w + 1) T / N), so the
// warps that share a (b, j) are consecutive and its partials can be numbered w + r (r = the
// (b, j) index; distinct for distinct segments): a contiguous run, which the combine finds
// from the requests' stream offsets (written to the workspace by the decode's first CTA).
#include <algorithm>
#include <mutex>

#include "combine_merge.cuh"
#include "paged_decode_mma.cuh"

namespace pkv {

namespace {

template <typename KV, int D, int G>
struct FlatShape {
  using M = MmaShape<KV, D, G, false>;
  static constexpr bool kFp8 = M::kFp8;
  static constexpr int kWarps = M::kWarps;
  static constexpr int kThreads = M::kThreads;
  static constexpr int NT = M::NT;
  static constexpr int SPW = M::SPW;
  static constexpr int STAGES = kWarps * SPW;
  static constexpr int BOXES = M::BOXES;
  static constexpr int BOX_ELEMS = M::BOX_ELEMS;
  static constexpr int TILE_BYTES = M::TILE_BYTES;
  static constexpr int STAGE_BYTES = M::STAGE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  // per warp: [G][D] values, [G] maxima, [G] sums, padded so that every warp's area starts
  // on a 16-byte boundary (its values are read as float4)
  static constexpr int WARP_FLOATS = G * D + (2 * G + 3) / 4 * 4;
  static constexpr int MERGE_BYTES = kWarps * WARP_FLOATS * 4;
  static constexpr int PT_BYTES = M::PT_BYTES;
  static constexpr int BAR_BYTES = STAGES * 8 + STAGES * 4;
  // bytes before the per-request page offsets ([batch + 1] ints follow)
  static constexpr int FIXED_BYTES =
      1024 + RING_BYTES + MERGE_BYTES + PT_BYTES + (BAR_BYTES + 15) / 16 * 16;
  static size_t smem_bytes(int batch) { return FIXED_BYTES + (size_t)(batch + 1) * 4; }
  static_assert(kWarps == kFlatWarpsPerCta, "the launch plan counts four warps per CTA");
};

__device__ __forceinline__ int flat_ctx(const DecodeArgs& a, int b) {
  return min(max(0, a.context_lens[b]), a.max_pages * kPageSize);
}

// The request whose pages hold stream page F: the last b with pre[b] * h_kv <= F (requests
// with no pages share their successor's offset and are never chosen).
__device__ __forceinline__ int flat_request(const int* pre, int batch, long long F, int h_kv) {
  const long long q = F / h_kv;
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Warp holding stream page P (of T, split over N warps): the last w with w T / N <= P.
__device__ __forceinline__ long long flat_owner(long long P, long long T, long long N) {
  return ((P + 1) * N + T - 1) / T - 1;
}

// (four CTAs per SM for narrow caches, as the chunked kernel gets; three for bf16, whose ring
// allows no more)
template <typename KV, typename TQ, int D, int G>
__global__ void __launch_bounds__(32 * PKV_MMA_WARPS, KV::bytes == 1 ? 4 : 3) paged_decode_flat_kernel(
    const DecodeArgs a, const int cap, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using S = FlatShape<KV, D, G>;
  constexpr bool F8 = S::kFp8;
  constexpr int NW = S::kWarps, SPW = S::SPW, NT = S::NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.batch, h_kv = a.h_kv;
  // the combine kernel (a programmatic dependent launch) may be scheduled once every CTA of
  // this grid has started; it waits for this grid's completion before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* red_acc = reinterpret_cast<float*>(smem + S::RING_BYTES) + warp * S::WARP_FLOATS;
  float* red_m = red_acc + G * D;
  float* red_l = red_m + G;
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + S::RING_BYTES + S::MERGE_BYTES) +
                 warp * NT * 8 * kPageSize;
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem + S::RING_BYTES + S::MERGE_BYTES + S::PT_BYTES);
  int* page_ok = reinterpret_cast<int*>(full + S::STAGES);
  int* pre = reinterpret_cast<int*>(smem + (S::FIXED_BYTES - 1024));  // [B + 1]

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  // pre[b] = pages the requests before b walk (per KV head): a scan over the block, each
  // thread taking a run of consecutive requests
  {
    __shared__ int warp_sum[NW];
    const int per = (B + S::kThreads - 1) / S::kThreads;
    const int b0 = threadIdx.x * per;
    int tot = 0;
    for (int k = 0; k < per; ++k) {
      const int b = b0 + k;
      if (b < B) {
        if (blockIdx.x == 0 && a.context_lens[b] > a.max_pages * kPageSize)
          atomicOr(a.err, PKV_DEVERR_BAD_PAGE);  // cut to the table width
        tot += seq_pages(flat_ctx(a, b), a.sink, a.window).n;
      }
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int run = incl - tot;
    for (int w = 0; w < warp; ++w) run += warp_sum[w];
    for (int k = 0; k < per; ++k) {
      const int b = b0 + k;
      if (b < B) {
        pre[b] = run;
        run += seq_pages(flat_ctx(a, b), a.sink, a.window).n;
      }
    }
    if (threadIdx.x == S::kThreads - 1) pre[B] = run;
    __syncthreads();
    if (blockIdx.x == 0)  // for the combine
      for (int b = threadIdx.x; b <= B; b += S::kThreads) a.flat_pre[b] = pre[b];
  }

  const long long T = (long long)pre[B] * h_kv;  // pages in the stream
  const long long N = (long long)gridDim.x * NW;
  const long long gw = (long long)blockIdx.x * NW + warp;
  const long long s0 = gw * T / N, s1 = (gw + 1) * T / N;  // this warp's share
  const int cap_g = cap;  // partial slots per head
  if (s0 >= s1) {
    // no pages: where this empty share sits inside a (b, j) (not at its start), the combine
    // counts it among that (b, j)'s partials -- leave an empty one
    if (s0 < T) {
      const int b = flat_request(pre, B, s0, h_kv);
      const int nb = pre[b + 1] - pre[b];
      const long long off = s0 - (long long)pre[b] * h_kv;
      const int j = (int)(off / nb), p = (int)(off % nb);
      if (p > 0) {
        const long long id = gw + (long long)b * h_kv + j;
        for (int g = 0; g < G; ++g) {
          const size_t part = (size_t)g * cap_g + id;
          for (int i = lane; i < D; i += 32) a.ws_acc[part * D + i] = 0.f;
          if (lane == 0) {
            a.ws_ml[part * 2] = -INFINITY;
            a.ws_ml[part * 2 + 1] = 0.f;
          }
        }
      }
    }
    return;
  }

  const uint64_t pol = l2_evict_first_policy();
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t pt_u32 = smem_u32(pt);
  const int n_mine = (int)(s1 - s0);

  // Pool row of each of the warp's pages, read 32 at a time ahead of their copies: lane L
  // holds the tile row of the warp's page 32 t + L (-1: its id is outside the pool).
  int rows = -1;
  auto load_rows = [&](int t) {
    const int mm = 32 * t + lane;
    rows = -1;
    if (mm < n_mine) {
      const long long F = s0 + mm;
      const int b = flat_request(pre, B, F, h_kv);
      const int nb = pre[b + 1] - pre[b];
      const long long off = F - (long long)pre[b] * h_kv;
      const int j = (int)(off / nb), p = (int)(off % nb);
      const SeqPages sp = seq_pages(flat_ctx(a, b), a.sink, a.window);
      const int pid = a.block_tables[(size_t)b * a.max_pages + logical_page(sp, p)];
      rows = (pid >= 0 && pid < a.num_pages) ? (pid * h_kv + j) * kPageSize : -1;
    }
  };
  auto issue = [&](int stg, int row) {  // lane 0: the tile at pool row `row` -> stage stg
    if (row < 0) {
      page_ok[stg] = 0;
      atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
      mbar_arrive(&full[stg]);
    } else {
      page_ok[stg] = 1;
      mbar_arrive_expect_tx(&full[stg], S::STAGE_BYTES);
      const uint32_t dst = ring_u32 + stg * S::STAGE_BYTES;
      tma_tile<S::BOXES, S::BOX_ELEMS>(dst, &tm_k, a.tma_rank, row, &full[stg], pol);
      tma_tile<S::BOXES, S::BOX_ELEMS>(dst + S::TILE_BYTES, &tm_v, a.tma_rank, row, &full[stg],
                                       pol);
    }
  };
  load_rows(0);
  {
    int first_rows[SPW];
#pragma unroll
    for (int m = 0; m < SPW; ++m) first_rows[m] = __shfl_sync(0xffffffffu, rows, m);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < SPW; ++m)
        if (m < n_mine) issue(warp * SPW + m, first_rows[m]);
    }
  }

  // the first segment: request b, KV head j, from its walked page p
  int b = flat_request(pre, B, s0, h_kv);
  int nb = pre[b + 1] - pre[b];
  int j, p;
  {
    const long long off = s0 - (long long)pre[b] * h_kv;
    j = (int)(off / nb);
    p = (int)(off % nb);
  }
  int m = 0;  // pages of the share attended so far (ring position)
  bool ok = true;
  while (m < n_mine) {
    const int ctx_in = max(0, a.context_lens[b]);
    const int ctx = min(ctx_in, a.max_pages * kPageSize);
    const SeqPages sp = seq_pages(ctx, a.sink, a.window);
    const int p_end = min(nb, p + (n_mine - m));  // (n_mine - m: pages left in the share)
    const int r = b * h_kv + j;
    // the segment holding the page of position ctx - 1 writes this step's rows there
    const bool appends = a.k_new != nullptr && p_end == nb && ctx == ctx_in && nb > 0;
    if (appends) append_prefetch<KV, D>(a, b, j, lane);
    MmaQuery<KV, TQ, D, G> Q;
    mma_load_query<KV, TQ, D, G>(a, b, j, lane, Q);
    MmaRun<D, G> R;
    R.reset();
    const int32_t* btrow = a.block_tables + (size_t)b * a.max_pages;
    for (int pp = p; pp < p_end; ++pp, ++m) {
      const int stg = warp * SPW + (m % SPW);
      const bool got = mbar_wait(&full[stg], (m / SPW) & 1, a.err);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      if (page_ok[stg]) {
        const int lp = logical_page(sp, pp);
        const int nvalid = min(kPageSize, ctx - lp * kPageSize);  // rows before the context end
        const uint32_t kt = ring_u32 + stg * S::STAGE_BYTES;
        const uint32_t vt = kt + S::TILE_BYTES;
        if (appends && pp == nb - 1) {
          uint8_t* ktp = ring + stg * S::STAGE_BYTES;
          fused_append_row<KV, D>(a, b, j, btrow[lp], nvalid - 1, ktp, ktp + S::TILE_BYTES, lane,
                                  [](int rr, int ch) { return (int)swz(rr, ch); });
          __syncwarp();
        }
        mma_attend_page<KV, TQ, D, G>(kt, vt, lp, nvalid, ctx, a.sink, a.window, Q, R, pt,
                                      pt_u32, lane);
      }
      __syncwarp();
      if (m + SPW < n_mine) {  // refill the stage with the share's page m + SPW (warp-uniform)
        const int mn = m + SPW;
        if ((mn & 31) == 0) load_rows(mn >> 5);
        const int row = __shfl_sync(0xffffffffu, rows, mn & 31);
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(stg, row);
        }
      }
    }
    if (!ok) break;

    // the segment's result: lane L owns dims 4L .. 4L+3 of every head
    mma_run_to_smem<KV, D, G>(R, red_acc, red_m, red_l, lane);
    __syncwarp();
    const float vs = F8 ? a.v_scales[j] : 1.f;
    const bool whole = p == 0 && p_end == nb;
    const long long id = gw + r;
    const int i0 = 4 * lane;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float Mg = red_m[g];
      const bool live = Mg != -INFINITY;
      const float Lg = live ? red_l[g] : 0.f;
      const float4 v = *reinterpret_cast<const float4*>(red_acc + g * D + i0);
      const float A[4] = {live ? v.x * vs : 0.f, live ? v.y * vs : 0.f, live ? v.z * vs : 0.f,
                          live ? v.w * vs : 0.f};
      if (whole) {
        const size_t o = ((size_t)b * a.h_q + j * G + g) * D + i0;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          store_from_float(static_cast<TQ*>(a.out), o + t, Lg > 0.f ? A[t] / Lg : 0.f);
      } else {
        const size_t part = (size_t)g * cap_g + id;
        *reinterpret_cast<float4*>(a.ws_acc + part * D + i0) = make_float4(A[0], A[1], A[2], A[3]);
        if (lane == 0) {
          a.ws_ml[part * 2] = Mg;
          a.ws_ml[part * 2 + 1] = Lg;
        }
      }
    }
    __syncwarp();  // the merge area is rewritten by the next segment
    // the next (b, j) of the stream
    p = p_end;
    if (p == nb) {
      p = 0;
      if (++j == h_kv) {
        j = 0;
        do {
          ++b;
        } while (b < B - 1 && pre[b + 1] == pre[b]);
      }
      nb = b < B ? pre[b + 1] - pre[b] : 0;
    }
  }
  if (!ok && lane == 0) {  // let the copies in flight land before the CTA's memory goes
    for (int mm = m; mm < n_mine && mm < m + SPW; ++mm)
      mbar_wait(&full[warp * SPW + (mm % SPW)], (mm / SPW) & 1, a.err);
  }
}

// The run of partials of (b, j) in the stream, from the page offsets the decode's first CTA
// wrote: nb pages per KV head; partial ids first + r .. first + r + count - 1.
__device__ __forceinline__ void flat_run(const DecodeArgs& a, int b, int j, int n_warps, int& nb,
                                         long long& first, int& count) {
  const int before = a.flat_pre[b], all = a.flat_pre[a.batch];
  nb = a.flat_pre[b + 1] - before;
  first = 0;
  count = 0;
  if (nb == 0) return;
  const long long T = (long long)all * a.h_kv, N = n_warps;
  const long long P0 = (long long)before * a.h_kv + (long long)j * nb;
  first = flat_owner(P0, T, N);
  count = (int)(flat_owner(P0 + nb - 1, T, N) - first + 1);
}

// Merges each (b, j)'s partials in stream order, once the decode grid is done (its run comes
// from the decode's page offsets); a (b, j) whose pages lie in one warp's share was written out
// by the decode (no partials), and one with no pages gets out = 0.
//  * PER_HEAD false (many (b, j), short runs): one CTA per (b, j); warp w merges heads w, w + 4,
//    ... one partial run each.
//  * PER_HEAD true (few (b, j), long runs): one CTA per (b, j, head g); the four warps merge a
//    quarter of the run each, then warp 0 merges the quarters in order.
template <typename TQ, int D, int G, bool PER_HEAD>
__global__ void __launch_bounds__(128) decode_flat_combine_kernel(const DecodeArgs a,
                                                                  const int cap,
                                                                  const int n_warps) {
  constexpr int DL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y, b = r / a.h_kv, j = r - b * a.h_kv;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid is done, its writes seen
  int nb, count;
  long long first;
  flat_run(a, b, j, n_warps, nb, first, count);
  if (count == 1) return;  // one warp's share holds the whole (b, j): the decode wrote out
  TQ* out = static_cast<TQ*>(a.out);
  if (!PER_HEAD) {
    for (int g = warp; g < G; g += 4) {
      const size_t o = ((size_t)b * a.h_q + j * G + g) * D + lane * DL;
      float M = -INFINITY, Lw = 0.f, A[DL];
#pragma unroll
      for (int k = 0; k < DL; ++k) A[k] = 0.f;
      if (count > 0) {
        const size_t part = (size_t)g * cap + (size_t)(first + r);
        merge_run<D, 8>(a.ws_ml + part * 2, a.ws_acc + part * D + lane * DL, 0, count, lane, M,
                        Lw, A);
      }
#pragma unroll
      for (int k = 0; k < DL; ++k) store_from_float(out, o + k, Lw > 0.f ? A[k] / Lw : 0.f);
    }
    return;
  }
  const int g = blockIdx.x;
  const size_t o = ((size_t)b * a.h_q + j * G + g) * D + lane * DL;
  if (count == 0) {  // no pages: out = 0 (the decode never writes this row)
    if (warp == 0)
#pragma unroll
      for (int k = 0; k < DL; ++k) store_from_float(out, o + k, 0.f);
    return;
  }
  const size_t part = (size_t)g * cap + (size_t)(first + r);
  __shared__ float red_a[4][D];
  __shared__ float red_ml[4][2];
  const int q = (count + 3) / 4;
  float M = -INFINITY, Lw = 0.f, A[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) A[k] = 0.f;
  merge_run<D, 8>(a.ws_ml + part * 2, a.ws_acc + part * D + lane * DL, min(count, warp * q),
                  min(count, (warp + 1) * q), lane, M, Lw, A);
#pragma unroll
  for (int k = 0; k < DL; ++k) red_a[warp][lane * DL + k] = A[k];
  if (lane == 0) {
    red_ml[warp][0] = M;
    red_ml[warp][1] = Lw;
  }
  __syncthreads();
  if (warp != 0) return;
  float Mw[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) Mw[w] = red_ml[w][0];
  M = fmaxf(fmaxf(Mw[0], Mw[1]), fmaxf(Mw[2], Mw[3]));
  Lw = 0.f;
#pragma unroll
  for (int k = 0; k < DL; ++k) A[k] = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {  // an empty quarter (maximum -inf) has weight 0
    const float sw = Mw[w] == -INFINITY ? 0.f : exp2f(Mw[w] - M);
    Lw = fmaf(sw, red_ml[w][1], Lw);
#pragma unroll
    for (int k = 0; k < DL; ++k) A[k] = fmaf(sw, red_a[w][lane * DL + k], A[k]);
  }
#pragma unroll
  for (int k = 0; k < DL; ++k) store_from_float(out, o + k, Lw > 0.f ? A[k] / Lw : 0.f);
}

// (b, j) rows below which the combine takes one CTA per head
constexpr int kFlatCombinePerHeadRows = 256;

template <typename KV, typename TQ, int D, int G>
struct FlatLaunch {
  // CTAs resident at once on the current device for this batch (one wave)
  static cudaError_t wave(int batch, int* ctas) {
    using S = FlatShape<KV, D, G>;
    auto kern = paged_decode_flat_kernel<KV, TQ, D, G>;
    const int smem = (int)S::smem_bytes(batch);
    // per device: the largest dynamic shared memory granted so far, and the wave of the last
    // size asked for (under a lock: callers may run on several host threads)
    constexpr int kDevs = 64;
    static int attr_smem[kDevs], occ_smem[kDevs], occ_ctas[kDevs];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (smem > attr_smem[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr_smem[dev] = smem;
    }
    if (smem != occ_smem[dev]) {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, S::kThreads, smem);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      occ_ctas[dev] = std::max(1, per_sm) * std::max(1, sms);
      occ_smem[dev] = smem;
    }
    *ctas = occ_ctas[dev];
    return cudaSuccess;
  }
  static cudaError_t decode(const DecodeArgs& a, int ctas, int cap, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s) {
    using S = FlatShape<KV, D, G>;
    int wv = 0;
    cudaError_t e = wave(a.batch, &wv);  // (sets the shared-memory attribute)
    if (e != cudaSuccess) return e;
    paged_decode_flat_kernel<KV, TQ, D, G><<<ctas, S::kThreads, S::smem_bytes(a.batch), s>>>(
        a, cap, tk, tv);
    return cudaGetLastError();
  }
  static cudaError_t combine(const DecodeArgs& a, int ctas, int cap, cudaStream_t s) {
    const int rows = a.batch * a.h_kv;
    const bool per_head = rows < kFlatCombinePerHeadRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(per_head ? G : 1, rows);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return per_head ? cudaLaunchKernelEx(&cfg, decode_flat_combine_kernel<TQ, D, G, true>, a,
                                         cap, ctas * kFlatWarpsPerCta)
                    : cudaLaunchKernelEx(&cfg, decode_flat_combine_kernel<TQ, D, G, false>, a,
                                         cap, ctas * kFlatWarpsPerCta);
  }
};

enum class FlatOp { kWave, kDecode, kCombine };

template <typename KV, typename TQ>
cudaError_t flat_g(FlatOp op, const DecodeArgs& a, int group, int* ctas, int cap,
                   const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
#define PKV_FLAT_CASE(GG)                                                             \
  case GG:                                                                            \
    if (op == FlatOp::kWave) return FlatLaunch<KV, TQ, 128, GG>::wave(a.batch, ctas); \
    if (op == FlatOp::kDecode)                                                        \
      return FlatLaunch<KV, TQ, 128, GG>::decode(a, *ctas, cap, tk, tv, s);          \
    return FlatLaunch<KV, TQ, 128, GG>::combine(a, *ctas, cap, s);
  switch (group) {
    PKV_FLAT_CASE(1)
    PKV_FLAT_CASE(2)
    PKV_FLAT_CASE(4)
    PKV_FLAT_CASE(8)
    PKV_FLAT_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef PKV_FLAT_CASE
}

cudaError_t flat_dispatch(FlatOp op, const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                          int* ctas, int cap, const void* tk, const void* tv, cudaStream_t s) {
  static const CUtensorMap none{};
  const CUtensorMap& k = tk ? *static_cast<const CUtensorMap*>(tk) : none;
  const CUtensorMap& v = tv ? *static_cast<const CUtensorMap*>(tv) : none;
  if (kv_dtype == PKV_BF16 && q_dtype == PKV_BF16)
    return flat_g<BF16, __nv_bfloat16>(op, a, group, ctas, cap, k, v, s);
  if (kv_dtype == PKV_FP8_E4M3 && q_dtype == PKV_BF16)
    return flat_g<FP8, __nv_bfloat16>(op, a, group, ctas, cap, k, v, s);
  if (kv_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F32)
    return flat_g<FP8, float>(op, a, group, ctas, cap, k, v, s);
  if (kv_dtype == PKV_INT8 && q_dtype == PKV_BF16)
    return flat_g<INT8, __nv_bfloat16>(op, a, group, ctas, cap, k, v, s);
  if (kv_dtype == PKV_INT8 && q_dtype == PKV_F32)
    return flat_g<INT8, float>(op, a, group, ctas, cap, k, v, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_flat_wave(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                             int* ctas) {
  return flat_dispatch(FlatOp::kWave, a, kv_dtype, q_dtype, group, ctas, 0, nullptr, nullptr,
                       nullptr);
}

cudaError_t launch_decode_flat(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                               int ctas, int cap, const void* tk, const void* tv,
                               cudaStream_t s) {
  return flat_dispatch(FlatOp::kDecode, a, kv_dtype, q_dtype, group, &ctas, cap, tk, tv, s);
}

cudaError_t launch_decode_flat_combine(const DecodeArgs& a, int kv_dtype, int q_dtype, int group,
                                       int ctas, int cap, cudaStream_t s) {
  return flat_dispatch(FlatOp::kCombine, a, kv_dtype, q_dtype, group, &ctas, cap, nullptr,
                       nullptr, s);
}

}  // namespace pkv
