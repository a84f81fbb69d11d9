// Shared-prefix pass of the cascade decode. Requests that start with the same prompt share
// its KV pages ("KV cache and PagedAttention", section 6: prefix caching reuses the pages of
// a common prefix; "KV Cache" glossary: a shared prompt's blocks serve several sequences).
// The plain decode reads those pages once per request; here one CTA reads a chunk of them
// once for up to 64 query rows of the group -- (member, query head) pairs of one KV head --
// which turns the group's Q.K^T and P.V into dense tensor-core contractions:
//
//  * rows: query rows of the group (M, 16 per warp), tokens of a page (N for the scores, K for
//    the values), head_dim (K for the scores, N for the values); mma.m16n8k16 bf16 -> fp32;
//  * staging: all warps share a ring of 4 stages of two pages each, the (page, KV head) K and
//    V tiles moved by 2-D TMA copies (128-byte swizzle) that complete on the stage's mbarrier;
//    a warp takes 32 tokens per step (two pages), which gives four independent MMA chains for
//    the scores and halves the softmax and rescaling work per token;
//  * scores S = Q K^T; the k order inside each 32-dim block is permuted so a lane's K operand
//    for two k-steps is one 16-byte shared load of its token's row, chosen so that the eight
//    lanes of each load phase hit eight different 16-byte bank groups; the queries use the
//    same permutation;
//  * base-2 online softmax per row (scores times scale * log2 e), with the probabilities kept
//    in registers as the A operand of P V (rounded to bf16); V fragments by ldmatrix.trans;
//  * each CTA writes its rows' partial (max, sum, weighted values) for its chunk of the prefix
//    to the chunk slots of every member; the members' own pages follow in later slots and the
//    combine kernel merges them all (the same partial-merge rule as the split decode).
#include <atomic>
#include <cuda.h>
#include <math.h>

#include "decode_plan.cuh"
#include "paged_decode_mma.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kCpRows = kCascadeRows;           // query rows per CTA
constexpr int kCpWarps = kCpRows / 16;          // 16 query rows per warp
constexpr int kCpStages = 4;                    // steps of two pages in flight per CTA
constexpr int kCpTile = kPageSize * 128 * 2;    // one (page, KV head) tile, bf16, d = 128
constexpr int kCpStage = 4 * kCpTile;           // K of two pages, then V of two pages
constexpr int kCpSmem = 1024 + kCpStages * kCpStage + kCpStages * 8 + 2 * kCpStages * 4;

// 16-byte chunk of a 256-byte bf16 row that lane `tig` reads for dim block kp (0..3): the 32
// dims of block kp are chunks kp0 .. with 2 tig + (kp & 1) + 8 (kp >> 1) covering each of the
// 16 chunks once over (kp, tig).
__device__ __forceinline__ int cp_chunk(int kp, int tig) {
  return 2 * tig + (kp & 1) + 8 * (kp >> 1);
}

template <int G>
__global__ void __launch_bounds__(32 * kCpWarps, 3) cascade_prefix_kernel(
    const DecodeArgs a, const CascadeArgs ca, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  constexpr int D = 128;
  const int c = blockIdx.x, rt = blockIdx.y;
  const int g = blockIdx.z / a.h_kv, j = blockIdx.z % a.h_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const bool reporter = c == 0 && rt == 0 && threadIdx.x == 0;
  // the own-page decode (a programmatic dependent launch) may start on the SMs this grid leaves
  // free; it waits for this grid's completion before it reads the partials written here
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int o0 = ca.group_offsets[g];
  int members = ca.group_offsets[g + 1] - o0;
  if (o0 < 0 || members < 0) {
    if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
    return;
  }
  if (members > ca.max_members) {
    if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
    members = ca.max_members;
  }
  const int n_rows = members * G;
  if (rt * kCpRows >= n_rows) return;
  if (a.prefix_pages[g] > a.max_prefix_pages && reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
  const int pp = cascade_group_pages(a, g);
  const int n_chunks = cascade_prefix_chunks(a, pp);
  if (c >= n_chunks) return;
  const int per_chunk = (pp + n_chunks - 1) / n_chunks;
  const int page0 = c * per_chunk;
  const int n_pages = max(0, min(per_chunk, pp - page0));
  // the group's shared pages: from the groups' id array, else as listed by its first member's
  // table row
  const int32_t* btrow;
  if (ca.prefix_ids != nullptr) {
    btrow = ca.prefix_ids + (size_t)g * ca.ids_stride;
  } else {
    const int b_first = ca.group_members[o0];
    if (b_first < 0 || b_first >= a.batch) {
      if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
      return;
    }
    btrow = a.block_tables + (size_t)b_first * a.max_pages;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kCpStages * kCpStage);
  int* page_ok = reinterpret_cast<int*>(full + kCpStages);  // [stage][2]
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCpStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  __syncthreads();

  const uint64_t pol = l2_evict_last_policy();  // every row tile of the group reads them
  const uint32_t smem_u = smem_u32(smem);
  const int n_steps = (n_pages + 1) / 2;
  auto issue = [&](int it, int stg) {  // thread 0: pages 2 it, 2 it + 1 into stage stg
    int bytes = 0;
    int pid[2];
    for (int k = 0; k < 2; ++k) {
      const int i = 2 * it + k;
      pid[k] = i < n_pages ? btrow[page0 + i] : -1;
      const bool ok = pid[k] >= 0 && pid[k] < a.num_pages;
      if (i < n_pages && !ok) atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
      page_ok[2 * stg + k] = ok;
      if (!ok) pid[k] = -1;
      bytes += ok ? 2 * kCpTile : 0;
    }
    if (bytes == 0) {
      mbar_arrive(&full[stg]);
      return;
    }
    mbar_arrive_expect_tx(&full[stg], bytes);
    const uint32_t dst = smem_u + stg * kCpStage;
    for (int k = 0; k < 2; ++k) {
      if (pid[k] < 0) continue;
      const int row = (pid[k] * a.h_kv + j) * kPageSize;
      tma_tile<2, 64>(dst + k * kCpTile, &tm_k, a.tma_rank, row, &full[stg], pol);
      tma_tile<2, 64>(dst + (2 + k) * kCpTile, &tm_v, a.tma_rank, row, &full[stg], pol);
    }
  };
  if (threadIdx.x == 0)
    for (int s = 0; s < kCpStages && s < n_steps; ++s) issue(s, s);

  // This warp's rows rt*64 + 16 warp + gid (+8): row r is query head j*G + r % G of request
  // group_members[o0 + r / G]. A fragments of Q for dim block kp, k order as cp_chunk.
  int rb[2], rh[2];
  bool live[2];
  uint4 qa[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = rt * kCpRows + warp * 16 + gid + 8 * h;
    live[h] = r < n_rows;
    rb[h] = live[h] ? ca.group_members[o0 + r / G] : 0;
    rh[h] = j * G + r % G;
    if (live[h] && (rb[h] < 0 || rb[h] >= a.batch)) {
      atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
      live[h] = false;
      rb[h] = 0;
    }
    const __nv_bfloat16* qrow =
        static_cast<const __nv_bfloat16*>(a.q) + ((size_t)rb[h] * a.h_q + rh[h]) * D;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp)
      qa[h][kp] = live[h] ? *reinterpret_cast<const uint4*>(qrow + 8 * cp_chunk(kp, tig))
                          : make_uint4(0, 0, 0, 0);
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  const float sc = a.scale_log2;
  const int lq = lane >> 3, lr = lane & 7;  // ldmatrix: matrix lq, row lr

  int it = 0;
  bool ok = true;
  for (; it < n_steps; ++it) {
    const int stg = it % kCpStages;
    const bool got = mbar_wait(&full[stg], (it / kCpStages) & 1, a.err);
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    const bool ok0 = page_ok[2 * stg] != 0, ok1 = page_ok[2 * stg + 1] != 0;  // CTA-uniform
    const uint32_t base = smem_u + stg * kCpStage;
    // ---- S[16 rows][32 tokens]: n-tile nt holds tokens 8 nt .. 8 nt + 7 ----
    float s[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      const int ch = cp_chunk(kp, tig);
      const uint4 x = qa[0][kp], y = qa[1][kp];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k == 0 ? !ok0 : !ok1) continue;
        const uint32_t kt = base + k * kCpTile;
        const uint4 k0 = lds128(kt + swz(gid, ch));
        const uint4 k8 = lds128(kt + swz(gid + 8, ch));
        mma16816<false>(s[2 * k], x.x, y.x, x.y, y.y, k0.x, k0.y);
        mma16816<false>(s[2 * k + 1], x.x, y.x, x.y, y.y, k8.x, k8.y);
        mma16816<false>(s[2 * k], x.z, y.z, x.w, y.w, k0.z, k0.w);
        mma16816<false>(s[2 * k + 1], x.z, y.z, x.w, y.w, k8.z, k8.w);
      }
    }
    // ---- online softmax; lane holds tokens 8 nt + 2 tig (+1) of rows gid (h = 0), gid+8 ----
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const bool v = (nt < 2) ? ok0 : ok1;
        s[nt][2 * h] = v ? s[nt][2 * h] * sc : -INFINITY;
        s[nt][2 * h + 1] = v ? s[nt][2 * h + 1] * sc : -INFINITY;
        mx = fmaxf(mx, fmaxf(s[nt][2 * h], s[nt][2 * h + 1]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[h] = exp2f(m_run[h] - m_use);
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        s[nt][2 * h] = exp2f(s[nt][2 * h] - m_use);
        s[nt][2 * h + 1] = exp2f(s[nt][2 * h + 1] - m_use);
        sum += s[nt][2 * h] + s[nt][2 * h + 1];
      }
      l_run[h] = l_run[h] * alpha[h] + sum;
      m_run[h] = m_new;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
    // ---- O[16 rows][128 dims] += P V, one 16-token k-step per page ----
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (k == 0 ? !ok0 : !ok1) continue;
      const uint32_t p0 = pack_bf16(s[2 * k][0], s[2 * k][1]);          // row gid, tokens 2tig..
      const uint32_t p1 = pack_bf16(s[2 * k][2], s[2 * k][3]);          // row gid+8
      const uint32_t p2 = pack_bf16(s[2 * k + 1][0], s[2 * k + 1][1]);  // row gid, tokens 8+2tig..
      const uint32_t p3 = pack_bf16(s[2 * k + 1][2], s[2 * k + 1][3]);  // row gid+8
      const uint32_t vt = base + (2 + k) * kCpTile;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vt + swz((lq & 1) * 8 + lr, 2 * mi + (lq >> 1)), b0, b1, b2, b3);
        mma16816<false>(o[2 * mi], p0, p1, p2, p3, b0, b1);
        mma16816<false>(o[2 * mi + 1], p0, p1, p2, p3, b2, b3);
      }
    }
    __syncthreads();  // every warp is done with stage stg
    if (threadIdx.x == 0 && it + kCpStages < n_steps) {
      fence_proxy_async_smem();
      issue(it + kCpStages, stg);
    }
  }
  if (!ok && threadIdx.x == 0) {  // let the copies still in flight land before leaving
    for (int k = it; k < n_steps && k < it + kCpStages; ++k)
      mbar_wait(&full[k % kCpStages], (k / kCpStages) & 1, a.err);
  }

  // ---- partials of this chunk for the warp's rows ----
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_run[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (!live[h]) continue;
    const size_t part = ((size_t)rb[h] * a.h_q + rh[h]) * a.n_chunk_slots + c;
    float* acc = a.ws_acc + part * D;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<float2*>(acc + 8 * nt + 2 * tig) = make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
    if (tig == 0) {
      a.ws_ml[part * 2 + 0] = m_run[h];
      a.ws_ml[part * 2 + 1] = l;
    }
  }
  if (!ok) __syncthreads();  // keep the CTA resident until the copies above have landed
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, const CascadeArgs& ca, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t s) {
  auto kern = cascade_prefix_kernel<G>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_done.load() >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCpSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done.fetch_or(1ull << dev);
  }
  const int chunks = (a.max_prefix_pages + a.prefix_chunk_pages - 1) / a.prefix_chunk_pages;
  const int tiles = (ca.max_members * G + kCpRows - 1) / kCpRows;
  dim3 grid(chunks, tiles, a.n_groups * a.h_kv);
  kern<<<grid, 32 * kCpWarps, kCpSmem, s>>>(a, ca, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cascade_prefix(const DecodeArgs& a, const CascadeArgs& ca, int group,
                                  const void* tk, const void* tv, cudaStream_t s) {
  const CUtensorMap& mk = *static_cast<const CUtensorMap*>(tk);
  const CUtensorMap& mv = *static_cast<const CUtensorMap*>(tv);
  switch (group) {
    case 1: return launch_g<1>(a, ca, mk, mv, s);
    case 2: return launch_g<2>(a, ca, mk, mv, s);
    case 4: return launch_g<4>(a, ca, mk, mv, s);
    case 8: return launch_g<8>(a, ca, mk, mv, s);
    case 16: return launch_g<16>(a, ca, mk, mv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
