// Single-token decode attention over a paged KV cache (the read phase of the KV-cache pages:
// the new token's query against every cached key and value, gathered through the request's
// page table -- "KV cache and PagedAttention", sections 1 and 4; GQA per the "KV Cache"
// glossary).
//
// One CTA = one (request b, KV head j, chunk c of up to chunk_pages pages). It serves the G
// query heads of the group, so each K/V tile is read from HBM once per group.
//
//  * Staging: every (page, KV head) tile of K and of V is one contiguous 16 x D block in the
//    pool. Each of the 4 warps owns SPW ring stages; its lane 0 fetches the warp's next pages
//    with 1-D bulk copies (cp.async.bulk, evict-first in L2) that complete on the stage's
//    mbarrier. Warp w consumes pages w, w+4, w+8, ... of the chunk, so while it computes one
//    page its next SPW-1 pages are in flight, and the CTA keeps 4*SPW pages in flight.
//  * Scores: lane L holds dims [L*DL, L*DL+DL) of the G query vectors (pre-multiplied by
//    scale*log2(e), and by the K scale for FP8) in registers. For a round of TOKR tokens
//    it forms TOKR*G partial dot products and reduces them across the warp with a
//    reduce-scatter butterfly of shuffles: each step halves the values a lane holds, so the
//    full reduction of NV values costs about NV shuffles instead of 5*NV.
//  * Online softmax (base 2): running max m and sum l per head, rescaled by exp2(m - m').
//  * Values: p values (and the rescale factors) go through a per-warp shared buffer; every
//    lane then accumulates p * V over its DL dims for all G heads.
//  * Merge: the 4 warps' (m, l, acc) are combined in shared memory. A single-chunk request
//    writes out = acc / l; otherwise the CTA writes its chunk's (m, l, acc) and the combine
//    kernel merges the chunks of each (b, h) in a fixed order. Chunk boundaries are logical
//    positions, so results do not depend on which physical pages hold the tokens.
#pragma once

#include <atomic>
#include <math.h>

#include "pkv_device.cuh"
#include "decode_epilogue.cuh"
#include "decode_plan.cuh"
#include "pkv_internal.h"

namespace pkv {

template <typename KV, int D, int G>
struct DecodeShape {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int DL = D / 32;                            // dims per lane
  static constexpr int TOKR = (16 * G <= 64) ? 16 : 64 / G;    // tokens per softmax round
  static constexpr int ROUNDS = kPageSize / TOKR;
  static constexpr int NV = TOKR * G;                          // partial sums per lane
  static constexpr int RS_STEPS = NV >= 32 ? 5 : (NV == 16 ? 4 : (NV == 8 ? 3 : 2));
  static constexpr int H = NV > 32 ? NV / 32 : 1;              // scores per lane after the RS
  static constexpr int DUP = 32 * H / NV;                      // lanes holding the same score
  static constexpr int RUN = 32 / G;                           // lanes holding one head's scores
  static constexpr int SPW = 2;                                // ring stages per warp
  static constexpr int STAGES = kWarps * SPW;
  static constexpr int ROW_BYTES = D * KV::bytes;
  static constexpr int TILE_BYTES = kPageSize * ROW_BYTES;
  static constexpr int RING_BYTES = STAGES * 2 * TILE_BYTES;
  static constexpr int MERGE_BYTES = kWarps * G * (D + 2) * 4;
  static constexpr int BIG_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int PB = (NV + G + 3) / 4 * 4;              // per-warp p + alpha floats
  static constexpr int SMEM_BYTES =
      BIG_BYTES + STAGES * 8 + STAGES * 4 + kWarps * PB * 4 + 16;
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(TOKR % 4 == 0, "tokens per round");
  static_assert(32 % G == 0, "group");
  static_assert((STAGES * 12) % 16 == 0, "per-warp buffers must stay 16-byte aligned");
};

// Reduce-scatter butterfly over 32 lanes: N values per lane in, N/2 after each step with a
// shuffle mask; once one value is left the remaining masks sum it across lanes.
template <int N, int MASK>
struct ReduceScatter {
  __device__ __forceinline__ static void run(float* v, int lane) {
    if constexpr (MASK == 0) {
      return;
    } else if constexpr (N >= 2) {
      const bool upper = (lane & MASK) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
      }
      ReduceScatter<N / 2, MASK / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
      ReduceScatter<1, MASK / 2>::run(v, lane);
    }
  }
};

template <int RUN>
__device__ __forceinline__ float run_max(float x) {
#pragma unroll
  for (int m = RUN / 2; m >= 1; m /= 2) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
  return x;
}

template <int RUN>
__device__ __forceinline__ float run_sum(float x) {
#pragma unroll
  for (int m = RUN / 2; m >= 1; m /= 2) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

template <typename KV, int D, int G>
struct WarpState {
  using S = DecodeShape<KV, D, G>;
  float m;              // running max (log2 domain) of this lane's head
  float l;              // this lane's share of the running sum
  float acc[G][S::DL];  // weighted values, all heads, this lane's dims
};

// One round of TOKR tokens of the page in shared memory (rows round*TOKR ..).
// Tokens: row r of the page is position tok0 + r; rows at or past nvalid lie beyond the
// context; win is (ctx, sink, window) for the attended-position test.
template <typename KV, int D, int G>
__device__ __forceinline__ void decode_round(WarpState<KV, D, G>& st,
                                             const float (&qf)[G][D / 32],
                                             const uint8_t* k_tile, const uint8_t* v_tile,
                                             int round, int nvalid, int tok0, int3 win, float* pb,
                                             int lane) {
  using S = DecodeShape<KV, D, G>;
  constexpr int DL = S::DL, TOKR = S::TOKR, NV = S::NV, H = S::H;
  float part[NV];
#pragma unroll
  for (int t = 0; t < TOKR; ++t) {
    float kf[DL];
    RowLoad<KV, DL>::run(k_tile + (round * TOKR + t) * S::ROW_BYTES + lane * DL * KV::bytes, kf);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < DL; ++i) a = fmaf(qf[g][i], kf[i], a);
      part[g * TOKR + t] = a;
    }
  }
  ReduceScatter<NV, 16>::run(part, lane);
  const int base = (lane >> (5 - S::RS_STEPS)) * H;  // index of this lane's first score
  const int gl = base / TOKR;
  float s[H];
  float mx = -INFINITY;
#pragma unroll
  for (int r = 0; r < H; ++r) {
    const int tok = round * TOKR + (base % TOKR) + r;
    s[r] = attended(tok0 + tok, win.x, win.y, win.z) ? part[r] : -INFINITY;
    mx = fmaxf(mx, s[r]);
  }
  mx = run_max<S::RUN>(mx);
  const float m_new = fmaxf(st.m, mx);
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
  const float alpha = exp2f(st.m - m_use);
  float psum = 0.f;
#pragma unroll
  for (int r = 0; r < H; ++r) {
    const float p = exp2f(s[r] - m_use);
    pb[base + r] = p;
    psum += p;
  }
  st.l = st.l * alpha + psum;
  st.m = m_new;
  if ((lane % S::RUN) == 0) pb[NV + gl] = alpha;
  __syncwarp();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float a = pb[NV + g];
#pragma unroll
    for (int i = 0; i < DL; ++i) st.acc[g][i] *= a;
  }
#pragma unroll
  for (int t0 = 0; t0 < TOKR; t0 += 4) {
    float4 p4[G];
#pragma unroll
    for (int g = 0; g < G; ++g) p4[g] = *reinterpret_cast<const float4*>(pb + g * TOKR + t0);
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int row = round * TOKR + t0 + tt;
      if (row < nvalid) {  // rows past the context may hold stale bytes (even NaN): skip them
        float vf[DL];
        RowLoad<KV, DL>::run(v_tile + row * S::ROW_BYTES + lane * DL * KV::bytes, vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = tt == 0 ? p4[g].x : tt == 1 ? p4[g].y : tt == 2 ? p4[g].z : p4[g].w;
#pragma unroll
          for (int i = 0; i < DL; ++i) st.acc[g][i] = fmaf(p, vf[i], st.acc[g][i]);
        }
      }
    }
  }
  __syncwarp();  // pb is rewritten by the next round
}

template <typename KV, typename TQ, int D, int G>
__global__ void __launch_bounds__(128) paged_decode_kernel(const DecodeArgs a) {
  using S = DecodeShape<KV, D, G>;
  constexpr int NW = S::kWarps, SPW = S::SPW, DL = S::DL, TILE = S::TILE_BYTES;
  const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int ctx = max(0, a.context_lens[b]);
  const bool cut = ctx > a.max_pages * kPageSize;
  if (cut) {  // longer than its page table: read what the table holds, append nothing
    if (c == 0 && threadIdx.x == 0) atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
    ctx = a.max_pages * kPageSize;
  }
  const SeqPlan plan = seq_plan(a, b, ctx);
  if (plan.prefix > 0 && ctx < plan.prefix * kPageSize + (a.k_new != nullptr ? 1 : 0)) {
    // a cascade member's context must reach past its group's shared pages
    if (c == 0 && threadIdx.x == 0) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
  }
  const SeqPages sp = plan.sp;
  const int pages_seq = sp.n;  // the pages read here, split into n_chunks near-equal chunks
  const int n_chunks = plan.n_chunks;
  // the combine kernel (a programmatic dependent launch) may be scheduled once every CTA of
  // this grid has started; it waits for this grid's completion before reading its partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (c > 0 && c >= n_chunks) return;
  const int per_chunk = n_chunks > 0 ? (pages_seq + n_chunks - 1) / n_chunks : 0;
  const int page0 = c * per_chunk;
  const int n_pages = max(0, min(per_chunk, pages_seq - page0));

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BIG_BYTES);
  int* page_ok = reinterpret_cast<int*>(full + S::STAGES);
  float* pbuf = reinterpret_cast<float*>(page_ok + S::STAGES) + warp * S::PB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  // this lane's slice of the group's queries, in the log2 domain
  float qf[G][DL];
  {
    const float qs = a.scale_log2 * (KV::bytes == 1 ? a.k_scales[j] : 1.f);
    const TQ* q = static_cast<const TQ*>(a.q);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < DL; ++i)
        qf[g][i] = load_as_float(q, ((size_t)b * a.h_q + j * G + g) * D + lane * DL + i) * qs;
  }

  const uint8_t* kc = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vc = static_cast<const uint8_t*>(a.v_cache);
  const int32_t* btrow = a.block_tables + (size_t)b * a.max_pages;
  const uint64_t pol = l2_evict_first_policy();

  auto issue = [&](int i, int stg, int pid) {  // lane 0: page i of the chunk (id pid) -> stage stg
    if (pid < 0 || pid >= a.num_pages) {
      page_ok[stg] = 0;
      atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
      mbar_arrive(&full[stg]);
    } else {
      page_ok[stg] = 1;
      mbar_arrive_expect_tx(&full[stg], 2 * TILE);
      const size_t off = ((size_t)pid * a.h_kv + j) * TILE;
      bulk_g2s(ring + stg * 2 * TILE, kc + off, TILE, &full[stg], pol);
      bulk_g2s(ring + stg * 2 * TILE + TILE, vc + off, TILE, &full[stg], pol);
    }
  };

  const int n_mine = n_pages > warp ? (n_pages - warp + NW - 1) / NW : 0;
  // Page ids of the warp's pages, read 32 at a time ahead of their copies so that no copy waits
  // on a table read: lane L holds the id of the warp's page 32 t + L (chunk page warp + NW m).
  int ids = -1;
  auto load_ids = [&](int t) {
    const int mm = 32 * t + lane;
    ids = mm < n_mine ? btrow[logical_page(sp, page0 + warp + NW * mm)] : -1;
  };
  load_ids(0);
  {
    int first[SPW];
#pragma unroll
    for (int m = 0; m < SPW; ++m) first[m] = __shfl_sync(0xffffffffu, ids, m);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < SPW; ++m)
        if (m < n_mine) issue(warp + NW * m, warp * SPW + m, first[m]);
    }
  }

  WarpState<KV, D, G> st;
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < DL; ++i) st.acc[g][i] = 0.f;

  int m = 0;
  bool ok = true;
  for (; m < n_mine; ++m) {
    const int i = warp + NW * m;
    const int stg = warp * SPW + (m % SPW);
    const bool got = mbar_wait(&full[stg], (m / SPW) & 1, a.err);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    if (page_ok[stg]) {
      const int lp = logical_page(sp, page0 + i);
      const int nvalid = min(kPageSize, ctx - lp * kPageSize);
      uint8_t* kt = ring + stg * 2 * TILE;
      if (a.k_new != nullptr && page0 + i == pages_seq - 1 && !cut) {
        fused_append_row<KV, D>(a, b, j, btrow[lp], nvalid - 1, kt, kt + TILE, lane,
                                [](int r, int ch) { return r * S::ROW_BYTES + 16 * ch; });
        __syncwarp();
      }
#pragma unroll 1
      for (int r = 0; r < S::ROUNDS; ++r)
        decode_round<KV, D, G>(st, qf, kt, kt + TILE, r, nvalid, lp * kPageSize,
                               make_int3(ctx, a.sink, a.window), pbuf, lane);
    }
    __syncwarp();
    if (m + SPW < n_mine) {  // warp-uniform
      const int mn = m + SPW;
      if ((mn & 31) == 0) load_ids(mn >> 5);
      const int pid = __shfl_sync(0xffffffffu, ids, mn & 31);
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(i + NW * SPW, stg, pid);
      }
    }
  }
  if (!ok && lane == 0) {
    // a wait gave up: wait (bounded) for this warp's copies still in flight before leaving
    for (int mm = m; mm < n_mine && mm < m + SPW; ++mm)
      mbar_wait(&full[warp * SPW + (mm % SPW)], (mm / SPW) & 1, a.err);
  }
  __syncthreads();  // all copies have landed: the ring is free for the merge

  float* red_acc = reinterpret_cast<float*>(ring);  // [NW][G][D]
  float* red_m = red_acc + NW * G * D;              // [NW][G]
  float* red_l = red_m + NW * G;                    // [NW][G]
  {
    const int base = (lane >> (5 - S::RS_STEPS)) * S::H;
    const int gl = base / S::TOKR;
    float lsum = run_sum<S::RUN>(st.l);
    if (S::DUP > 1) lsum *= 1.0f / S::DUP;
    if ((lane % S::RUN) == 0) {
      red_m[warp * G + gl] = st.m;
      red_l[warp * G + gl] = lsum;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < DL; ++i) red_acc[(warp * G + g) * D + lane * DL + i] = st.acc[g][i];
  }
  __syncthreads();

  const float vs = KV::bytes == 1 ? a.v_scales[j] : 1.f;
  decode_epilogue<TQ, D, G, NW, S::kThreads>(a, b, j, c, n_chunks, plan.slot0, red_acc,
                                             red_m, red_l, vs);
}

template <typename KV, typename TQ, int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  using S = DecodeShape<KV, D, G>;
  auto kern = paged_decode_kernel<KV, TQ, D, G>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device, per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_done.load() >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done.fetch_or(1ull << dev);
  }
  dim3 grid(a.chunk_grid, a.h_kv, a.batch);
  kern<<<grid, S::kThreads, S::SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

template <typename KV, typename TQ, int D>
cudaError_t launch_decode_g(const DecodeArgs& a, int group, cudaStream_t s) {
  switch (group) {
    case 1: return launch_decode_t<KV, TQ, D, 1>(a, s);
    case 2: return launch_decode_t<KV, TQ, D, 2>(a, s);
    case 4: return launch_decode_t<KV, TQ, D, 4>(a, s);
    case 8: return launch_decode_t<KV, TQ, D, 8>(a, s);
    case 16: return launch_decode_t<KV, TQ, D, 16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename KV, typename TQ>
cudaError_t launch_decode_d(const DecodeArgs& a, int head_dim, int group, cudaStream_t s) {
  if (head_dim == 64) return launch_decode_g<KV, TQ, 64>(a, group, s);
  if (head_dim == 128) return launch_decode_g<KV, TQ, 128>(a, group, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
