// Shared-prefix pass of the cascade decode on the fifth-generation tensor cores (tcgen05).
//
// Same result as the mma.sync prefix kernel (cascade_prefix.cu): for 128 query rows -- the
// (member, query head) pairs of one KV head of one group -- and a chunk of the group's shared
// pages ("KV cache and PagedAttention", section 6), the partial (max, sum, weighted values) of
// softmax attention over those pages. Here the two contractions run as tcgen05 MMAs whose A
// operands and accumulators live in tensor memory, so that the tensor core fetches only K and
// V from shared memory (with Q and P in shared memory too, ncu showed the tcgen05 pipe ~80 %
// busy on operand fetches while its math ran ~45 % of the time):
//
//  * a copy warp (lane 0) streams 64-token tiles (4 pages) of K and V into a 6-stage ring with
//    TMA copies (128-byte swizzle), refilling a stage as soon as the P V of its tile is done;
//    an MMA warp (lane 0) issues the MMAs:
//      S = Q K^T   M = 128 rows, N = 64 tokens, K = 128 dims  (8 MMAs of K = 16), S in TMEM;
//      O += P V    M = 128 rows, N = 128 dims, K = 16 tokens (a page): 4 MMAs, O in TMEM;
//    Q (A of S) and P (A of P V) are read from TMEM; K arrives as two swizzled
//    [64 rows][64 dims] blocks (2-D boxes, two per page), K-major; V as one 4 KB block per page
//    (a 3-D box), an MN-major operand;
//  * four softmax warps, one per TMEM lane quarter, so thread r owns row r: it writes its query
//    row into TMEM and zeroes its row of O once, then per tile reads its row of S
//    (tcgen05.ld), applies the scale (log2 domain), writes P = exp2(s - m) as bf16 pairs over
//    the first half of the same TMEM columns and keeps the row sum in a register;
//  * S (then P) has three TMEM buffers: the MMA warp keeps S up to three tiles ahead of the
//    softmax, and the P V of tile t overlaps the softmax of tile t+1; S(t+3) is issued only
//    once the P V of tile t, which reads P(t) from that buffer, has completed;
//  * the running maximum is updated lazily: O (in TMEM) is rescaled only when a row's maximum
//    grows by more than 2^8 (until then P <= 2^8), so most tiles never touch O; the final
//    (max, sum, O) triple is exact whatever maximum it was accumulated against.
//
// The query rows are read by the row threads while tensor memory is allocated and the first
// copies start; each row's partial leaves through shared memory and one bulk copy.
// Every wait is bounded (PKV_DEVERR_TIMEOUT); the TMEM columns are freed on every exit path.
#include <atomic>
#include <cuda.h>
#include <math.h>

#include "decode_plan.cuh"
#include "paged_decode_mma.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kTcRows = kCascadeTcRows;                  // query rows per CTA (MMA M)
constexpr int kTcSoftWarps = kTcRows / 32;               // one per TMEM lane quarter
constexpr int kTcMmaWarp = kTcSoftWarps;                 // issues the MMAs (lane 0)
constexpr int kTcCopyWarp = kTcSoftWarps + 1;            // issues the TMA copies (lane 0)
constexpr int kTcThreads = 32 * (kTcSoftWarps + 2);
constexpr int kTcTok = 64;                               // tokens per tile
constexpr int kTcPages = kTcTok / kPageSize;             // pages per tile
constexpr int kTcStages = 6;
constexpr int kTcKV = kTcTok * 256;                      // K (or V) of one tile
constexpr int kTcStageBytes = 2 * kTcKV;
constexpr int kTcOffBar = kTcStages * kTcStageBytes;
constexpr int kTcSmem = 1024 + kTcOffBar + 256;
static_assert(kTcSmem <= 227 * 1024, "shared memory of one CTA");
static_assert(8 * (2 * kTcStages + 3 + 3 + 2) + 4 * kTcStages + 4 <= 256, "barrier area");
static_assert(kTcRows * 528 <= kTcOffBar, "partial staging over the ring");
constexpr int kTcSBufs = 3;                              // S (then P) buffers in TMEM
// tensor memory columns: O [0, 128), Q [128, 192) (bf16 pairs), S buffer b at 192 + 64 b; P
// (bf16 pairs) overwrites the first 32 columns of its tile's S buffer
constexpr uint32_t kTcColQ = 128;
constexpr uint32_t kTcColS = 192;
constexpr uint32_t kTcTmemCols = 512;
static_assert(kTcColS + 64 * kTcSBufs <= kTcTmemCols, "tensor memory columns");
constexpr float kTcLazyLog2 = 8.f;

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major or MN-major, shape M x N.
constexpr uint32_t tc_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescS = tc_idesc(kTcRows, kTcTok, false);
constexpr uint32_t kIdescPV = tc_idesc(kTcRows, 128, true);

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading-dimension byte
// offset, stride byte offset (8-row groups), descriptor version 1.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// D (+)= A B with the A operand in tensor memory (its 128 lanes are A's rows; its 32-bit columns
// hold bf16 pairs along K, the lower index in the low half) and B described in shared memory.
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The barrier gets one arrival when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32 (w % 4) ..).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x with the special-function unit's approximation (relative error about 2^-22; results
// below 2^-126 flush to zero). The softmax arguments here are at most 2^8 (lazy rescaling) and
// P is rounded to bf16 right after, so the full-range exp2f buys nothing (measured: 1.8 us of
// a 26.6 us prefix pass on the prefix-sharing layer).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) cascade_prefix_tc_kernel(
    const DecodeArgs a, const CascadeArgs ca, const __grid_constant__ CUtensorMap tm_k2,
    const __grid_constant__ CUtensorMap tm_v) {
  constexpr int D = 128;
  constexpr int NS = kTcStages, SB = kTcSBufs;
  const int c = blockIdx.x, rt = blockIdx.y;
  const int g = blockIdx.z / a.h_kv, j = blockIdx.z % a.h_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool reporter = c == 0 && rt == 0 && threadIdx.x == 0;
  // the own-page decode (a programmatic dependent launch) may start on the SMs this grid leaves
  // free; it waits for this grid's completion before it reads the partials written here
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- the CTA's rows and pages (uniform exits before any barrier) ----
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
  if (rt * kTcRows >= n_rows) return;
  if (a.prefix_pages[g] > a.max_prefix_pages && reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
  const int pp = cascade_group_pages(a, g);
  const int n_chunks = cascade_prefix_chunks(a, pp);
  if (c >= n_chunks) return;
  const int per_chunk = (pp + n_chunks - 1) / n_chunks;
  const int page0 = c * per_chunk;
  const int n_pages = max(0, min(per_chunk, pp - page0));
  const int n_tiles = (n_pages + kTcPages - 1) / kTcPages;
  if (n_tiles == 0) return;
  // the chunk's page ids: from the groups' id array (one read), else from the first member's
  // table row (member, then row)
  const int32_t* idrow;
  if (ca.prefix_ids != nullptr) {
    idrow = ca.prefix_ids + (size_t)g * ca.ids_stride;
  } else {
    const int b_first = ca.group_members[o0];
    if (b_first < 0 || b_first >= a.batch) {
      if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
      return;
    }
    idrow = a.block_tables + (size_t)b_first * a.max_pages;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_u = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcOffBar);  // [NS]
  uint64_t* o_done = full + NS;                                     // [NS]: P V of a tile
  uint64_t* s_done = o_done + NS;                                   // [SB]
  // [SB]: P of a tile written (one per S buffer: the softmax warps can be up to SB - 1 tiles
  // apart, since S(t + SB) waits for the P V of tile t, so no warp arrives for tile t + SB
  // before the barrier of tile t has completed)
  uint64_t* p_ready = s_done + SB;
  uint64_t* q_ready = p_ready + SB;                                 // [1]
  uint64_t* mma_idle = q_ready + 1;                                 // [1]
  int* page_mask = reinterpret_cast<int*>(mma_idle + 1);            // [NS]
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(page_mask + NS);

  // The row threads read their query rows (two dependent reads: member id, then the row)
  // while the MMA warp allocates tensor memory and the copy warp starts the first copies.
  const int r = threadIdx.x;  // row of a softmax thread
  const int R = rt * kTcRows + r;
  bool live = false;
  int rb = 0;
  const int rh = j * G + R % G;
  uint4 qv[16];
  if (warp < kTcSoftWarps) {
    live = R < n_rows;
    rb = live ? ca.group_members[o0 + R / G] : 0;
    if (live && (rb < 0 || rb >= a.batch)) {
      atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
      live = false;
      rb = 0;
    }
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                       ((size_t)rb * a.h_q + rh) * D);
#pragma unroll
    for (int c16 = 0; c16 < 16; ++c16) qv[c16] = live ? qrow[c16] : make_uint4(0, 0, 0, 0);
  } else if (warp == kTcMmaWarp) {  // the TMEM columns: O, Q and the S buffers
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_taddr)),
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else if (lane == 0) {  // copy warp
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&o_done[s], 1);
    }
    for (int s = 0; s < SB; ++s) mbar_init(&s_done[s], 1);
    for (int s = 0; s < SB; ++s) mbar_init(&p_ready[s], kTcRows);
    mbar_init(q_ready, kTcRows);
    mbar_init(mma_idle, 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k2)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  const uint64_t pol = l2_evict_last_policy();  // every row tile of the group reads them
  // Copy warp: lane L holds the id of chunk page 32 m + L for the current batch m of 8 tiles,
  // read ahead of the copies so that no copy waits on a table read.
  int ids = -1;
  auto load_ids = [&](int m) {
    const int i = 32 * m + lane;
    ids = i < n_pages ? idrow[page0 + i] : -1;
  };
  auto issue = [&](int t, int st) {  // copy warp, all lanes: tile t into stage st
    if ((t & 7) == 0) load_ids(t >> 3);
    int pid[kTcPages];
#pragma unroll
    for (int p = 0; p < kTcPages; ++p) pid[p] = __shfl_sync(0xffffffffu, ids, (4 * t + p) & 31);
    if (lane != 0) return;
    int mask = 0, fill = 0;
    for (int p = 0; p < kTcPages; ++p) {
      if (t * kTcPages + p >= n_pages) {
        pid[p] = -1;
      } else if (pid[p] < 0 || pid[p] >= a.num_pages) {
        atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
        pid[p] = -1;
      } else {
        if (!mask) fill = pid[p];
        mask |= 1 << p;
      }
    }
    // A masked slot (past the chunk, or a bad id) gets a copy of a valid page of the tile:
    // its P is 0 and must meet finite V values. A tile with no valid page skips P V.
    int rows[kTcPages];
    for (int p = 0; p < kTcPages; ++p)
      rows[p] = ((pid[p] >= 0 ? pid[p] : fill) * a.h_kv + j) * kPageSize;
    page_mask[st] = mask;
    mbar_arrive_expect_tx(&full[st], kTcStageBytes);  // releases page_mask
    const uint32_t dst = stage_u + st * kTcStageBytes;
    for (int p = 0; p < kTcPages; ++p) {
      // K: the tile's 64 rows as two swizzled blocks of [64 rows][64 dims] (page p's rows at
      // p * 2048 in each), the layout of one N = 64 operand
      for (int bx = 0; bx < 2; ++bx)
        tma_load_2d(dst + bx * (kTcKV / 2) + p * 2048, &tm_k2, bx * 64, rows[p], &full[st], pol);
      // V: page p as one 4 KB block (two [16 rows][64 dims] halves), one K = 16 step of P V
      tma_tile<2, 64>(dst + kTcKV + p * 4096, &tm_v, a.tma_rank, rows[p], &full[st], pol);
    }
  };
  int issued = 0;
  if (warp == kTcCopyWarp) {
    __syncwarp();  // lane 0 initialised the barriers
    for (; issued < NS && issued < n_tiles; ++issued) issue(issued, issued);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_taddr;
  const float sc = a.scale_log2;

  if (warp == kTcCopyWarp) {
    // ===================== copy warp (lane 0 issues the copies) =====================
    // refill the stage of tile t with tile t + NS once the P V of tile t is done
    for (int t = 0; issued < n_tiles; ++t, ++issued) {
      const bool got = mbar_wait(&o_done[t % NS], (t / NS) & 1, a.err);
      if (!__all_sync(0xffffffffu, got)) break;
      issue(issued, issued % NS);
    }
    if (lane == 0) {  // before leaving, every copy issued has landed
      for (int t = max(0, issued - NS); t < issued; ++t)
        mbar_wait(&full[t % NS], (t / NS) & 1, a.err);
    }
  } else if (warp == kTcMmaWarp) {
    // ===================== MMA warp (lane 0) =====================
    if (lane == 0) {
      bool ok = mbar_wait(q_ready, 0, a.err);  // Q stored in TMEM and O zeroed
      tc_fence_after();
      auto pv = [&](int u) {  // O += P(u) V(u), P read from its tile's S buffer in TMEM
        if (!mbar_wait(&p_ready[u % SB], (u / SB) & 1, a.err)) return false;
        tc_fence_after();
        const int st = u % NS;
        const uint32_t vb = stage_u + st * kTcStageBytes + kTcKV;
        const uint32_t p_tmem = tmem + kTcColS + 64 * (u % SB);
        if (page_mask[st] != 0) {  // O starts at zero (stored by the row threads)
#pragma unroll
          for (int kk = 0; kk < kTcTok / 16; ++kk)
            tc_mma_ta(tmem, p_tmem + 8 * kk, tc_desc(vb + kk * 4096, 2048, 1024), kIdescPV, 1u);
        }
        tc_commit(&o_done[st]);
        return true;
      };
      auto s_mma = [&](int t) {  // S(t) = Q K(t)^T into S buffer t % SB, Q read from TMEM
        const int st = t % NS;
        if (!mbar_wait(&full[st], (t / NS) & 1, a.err)) return false;
        tc_fence_after();
        const uint32_t kb = stage_u + st * kTcStageBytes;
        const uint32_t s_tmem = tmem + kTcColS + 64 * (t % SB);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ta(s_tmem, tmem + kTcColQ + 8 * kk,
                    tc_desc(kb + (kk >> 2) * (kTcKV / 2) + (kk & 3) * 32, 16, 1024), kIdescS,
                    kk > 0 ? 1u : 0u);
        tc_commit(&s_done[t % SB]);
        return true;
      };
      // S runs up to SB tiles ahead of P V. S(u + SB) overwrites the buffer that P(u) lives in,
      // so it is issued only once the P V of tile u has completed.
      for (int t = 0; ok && t < SB && t < n_tiles; ++t) ok = s_mma(t);
      for (int u = 0; ok && u < n_tiles; ++u) {
        ok = pv(u);
        if (ok && u + SB < n_tiles) {
          ok = mbar_wait(&o_done[u % NS], (u / NS) & 1, a.err);
          if (ok) ok = s_mma(u + SB);
        }
      }
      // before leaving, every MMA issued is complete (on every path)
      tc_commit(mma_idle);
      mbar_wait(mma_idle, 0, a.err);
    }
  } else {
    // ===================== softmax warps: thread r owns row r =====================
    const uint32_t lane_t = tmem + ((uint32_t)(warp * 32) << 16);
    {  // Q into its TMEM columns (bf16 pairs along the head dimension), O = 0
      uint32_t w[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w[4 * k] = qv[8 * h + k].x;
          w[4 * k + 1] = qv[8 * h + k].y;
          w[4 * k + 2] = qv[8 * h + k].z;
          w[4 * k + 3] = qv[8 * h + k].w;
        }
        tmem_st32(lane_t + kTcColQ + 32 * h, w);
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = 0u;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) tmem_st32(lane_t + 32 * cb, w);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    float m_used = -INFINITY, l = 0.f;
    int t = 0;
    bool ok = true;
    for (; t < n_tiles; ++t) {
      const int st = t % NS;
      ok = mbar_wait(&full[st], (t / NS) & 1, a.err) &&
           mbar_wait(&s_done[t % SB], (t / SB) & 1, a.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int mask = page_mask[st];
      tc_fence_after();
      uint32_t sr[64];
      const uint32_t s_col = kTcColS + 64 * (t % SB);
      tmem_ld32(lane_t + s_col, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(lane_t + s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      if (mask != (1 << kTcPages) - 1) {  // masked pages score -inf
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (!((mask >> (k >> 4)) & 1)) sr[k] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], __uint_as_float(sr[k]));
      const float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float mx = mraw * sc;  // the scale is positive: max commutes with it
      if (t == 0) {
        m_used = mx;
      } else {
        const bool need = mx > m_used + kTcLazyLog2;
        if (__any_sync(0xffffffffu, need)) {  // rescale this warp's rows of O (in TMEM)
          const int u = t - 1;
          ok = mbar_wait(&o_done[u % NS], (u / NS) & 1, a.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float m_new = need ? mx : m_used;
          const float alpha = exp2f(m_used - m_new);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t o[32];
            tmem_ld32(lane_t + 32 * cb, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(lane_t + 32 * cb, o);
          }
          tmem_wait_st();
          l *= alpha;
          m_used = m_new;
        }
      }
      // P = 2^(s - m) as bf16 pairs over the first 32 columns of the tile's S buffer (its S
      // is in registers now); the P V MMA reads it from there
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pw[32];
      float sum8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sum8[k] = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * k]), sc, -m_use));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * k + 1]), sc, -m_use));
        sum8[(2 * k) & 7] += p0;
        sum8[(2 * k + 1) & 7] += p1;
        pw[k] = pack_bf16(p0, p1);
      }
      tmem_st32(lane_t + s_col, pw);
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[t % SB]);
    }
    // ---- the row's partial for this chunk ----
    if (ok) {
      const int u = n_tiles - 1;
      ok = mbar_wait(&o_done[u % NS], (u / NS) & 1, a.err);
    }
    if (__all_sync(0xffffffffu, ok)) {
      // every MMA and copy of the CTA is complete: the row's O goes through shared memory (the
      // free ring, rows 528 bytes apart: no bank conflicts), then one bulk copy of its 512
      // bytes to the workspace
      tc_fence_after();
      const uint32_t orow = stage_u + r * 528;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t o[32];
        tmem_ld32(lane_t + 32 * cb, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          sts128(orow + cb * 128 + k * 16, make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]));
      }
      if (live) {
        const size_t part = ((size_t)rb * a.h_q + rh) * a.n_chunk_slots + c;
        fence_proxy_async_smem();
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 512;" ::"l"(
                         a.ws_acc + part * D),
                     "r"(orow)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        a.ws_ml[part * 2 + 0] = m_used;
        a.ws_ml[part * 2 + 1] = l;
        // the shared-memory source is read before the CTA exits (the global writes complete
        // with the grid)
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTcTmemCols)
                 : "memory");
  }
}

template <int G>
cudaError_t launch_tc_g(const DecodeArgs& a, const CascadeArgs& ca, const CUtensorMap& tk,
                        const CUtensorMap& tv, cudaStream_t s) {
  auto kern = cascade_prefix_tc_kernel<G>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_done.load() >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done.fetch_or(1ull << dev);
  }
  const int chunks = (a.max_prefix_pages + a.prefix_chunk_pages - 1) / a.prefix_chunk_pages;
  const int tiles = (ca.max_members * G + kTcRows - 1) / kTcRows;
  dim3 grid(chunks, tiles, a.n_groups * a.h_kv);
  kern<<<grid, kTcThreads, kTcSmem, s>>>(a, ca, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cascade_prefix_tc(const DecodeArgs& a, const CascadeArgs& ca, int group,
                                     const void* tk, const void* tv, cudaStream_t s) {
  const CUtensorMap& mk = *static_cast<const CUtensorMap*>(tk);
  const CUtensorMap& mv = *static_cast<const CUtensorMap*>(tv);
  switch (group) {
    case 1: return launch_tc_g<1>(a, ca, mk, mv, s);
    case 2: return launch_tc_g<2>(a, ca, mk, mv, s);
    case 4: return launch_tc_g<4>(a, ca, mk, mv, s);
    case 8: return launch_tc_g<8>(a, ca, mk, mv, s);
    case 16: return launch_tc_g<16>(a, ca, mk, mv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
