// Single-token paged decode attention on tensor cores (bf16, FP8 E4M3 or INT8 cache,
// head_dim 128).
//
// Same computation, work split and results contract as paged_decode.cuh (the read phase of the
// KV-cache pages, "KV cache and PagedAttention" sections 1 and 4, GQA per the "KV Cache"
// glossary); what changes is how a warp turns one 16-token page into scores and weighted
// values. On CUDA cores that takes ~1260 instructions per 8 KiB page (shuffle reductions,
// per-element widening and FMAs) and the kernel is issue-bound; here it is ~16 tensor-core
// MMAs plus a few dozen other instructions per page.
//
//  * Staging: TMA tensor copies (128-byte swizzle) move each (page, KV head) tile of K and of
//    V into a warp-owned ring stage, completing on the stage's mbarrier: a bf16 pool is viewed
//    as a 3-D tensor [2 halves][rows][64 dims], so one box moves a whole 4 KiB tile as two
//    swizzled blocks; FP8/INT8 rows of 128 bytes take one 2-D box. The swizzle makes the
//    fragment loads below free of shared-memory bank conflicts. Each warp reads the page ids
//    of its pages 32 at a time (one per lane) ahead of their copies.
//  * Scores: S^T = K Q^T with mma.m16n8k16 -- the page's 16 tokens are M, the group's query
//    heads (padded to 8 per n-tile) are N, head_dim is K. The k order inside each 16-wide
//    k-step is permuted so a lane's A fragment for two k-steps is one 16-byte load of its row;
//    the query fragments (held in registers for the whole CTA) use the same permutation.
//  * Online softmax (base 2) on the accumulator fragment: a lane holds 2 tokens x 2 heads;
//    the page max per head needs 3 shuffles.
//  * Values: O^T = V^T P^T with mma.m16n8k16 -- head_dim is M (8 m-tiles), heads are N, the
//    page's tokens are K. V^T fragments come from ldmatrix.trans on the swizzled tile; P is
//    rounded to the MMA input type and transposed through a 256-byte per-warp buffer.
//  * FP8 / INT8: codes are widened to f16 in registers, four per 32-bit word (K fragments
//    from 16-byte loads; V^T fragments by pairing the codes of consecutive tokens with byte
//    permutes), the query is used in f16, and the MMAs run in f16 with fp32 accumulation; the
//    K scale multiplies the scores and the V scale the output. The widening is exact, except
//    that INT8 codes carry a bias: the softmax cancels it in the scores (widen4_scores), and
//    in the weighted values it comes off once per head at the end (MmaRun).
//  * Fused append: the CTA that reads the page holding position ctx-1 writes this step's K/V
//    row into the pool and into its staged copy of the page first (decode_epilogue.cuh).
//  * Rows of the last page past the context may hold stale bytes (even NaN): their scores are
//    set to -inf and their V rows to zero before the P.V product.
#pragma once

#include <atomic>
#include <cuda.h>
#include <math.h>

#include "pkv_device.cuh"
#include "decode_epilogue.cuh"
#include "decode_plan.cuh"
#include "pkv_internal.h"

namespace pkv {

#ifndef PKV_MMA_WARPS
#define PKV_MMA_WARPS 4  // warps per CTA
#endif
#ifndef PKV_MMA_SPW
#define PKV_MMA_SPW 2  // ring stages per warp
#endif

template <typename KV, int D, int G, bool WU = false>
struct MmaShape {
  static_assert(D == 128, "tensor-core decode supports head_dim 128");
  static constexpr bool kFp8 = KV::bytes == 1;
  static constexpr int kWarps = PKV_MMA_WARPS;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int NT = (G + 7) / 8;                 // n-tiles of 8 query heads
  static constexpr int KP = D / 32;                      // pairs of 16-wide k-steps
  static constexpr int MT = D / 16;                      // m-tiles of the P.V product
  // ring stages per warp: a warp that streams a whole short request keeps three copies in
  // flight (twelve stages per CTA, still one wave at two CTAs per SM)
  static constexpr int SPW = WU ? 3 : PKV_MMA_SPW;
  static constexpr int STAGES = kWarps * SPW;
  static constexpr int ROW_BYTES = D * KV::bytes;        // 256 (bf16) or 128 (fp8)
  static constexpr int BOXES = ROW_BYTES / 128;          // 128-byte swizzle boxes per row
  static constexpr int BOX_ELEMS = 128 / KV::bytes;
  static constexpr int TILE_BYTES = kPageSize * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int PT_BYTES = kWarps * NT * 8 * kPageSize * 2;          // P^T buffers
  static constexpr int MERGE_BYTES = kWarps * G * (D + 2) * 4;
  // the merge area aliases the ring, except with one warp per request (warps finish apart)
  static constexpr int BIG_BYTES =
      ((WU ? RING_BYTES + MERGE_BYTES : (RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES)) +
       1023) / 1024 * 1024;
  static constexpr int SMEM_BYTES =
      1024 + BIG_BYTES + PT_BYTES + STAGES * 8 + STAGES * 4;
};

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3, uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    mma16816_f16(d, a0, a1, a2, a3, b0, b1);
  else
    mma16816_bf16(d, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`; L2 evict-first.
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map, int x,
                                            int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled TMA load of one box (a whole (page, KV head) tile of a bf16 pool, as two
// swizzled 2 KB blocks: the first 64 dims of its 16 rows, then the last 64).
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const CUtensorMap* map, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// One (page, KV head) tile of K or V into shared memory: one 3-D box for a bf16 pool whose
// tensor map has rank 3, else one 2-D box per 128 bytes of row.
template <int BOXES, int BOX_ELEMS>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, int rank, int row,
                                         uint64_t* bar, uint64_t policy) {
  if (BOXES == 2 && rank == 3) {
    tma_load_3d(dst, map, row, bar, policy);
  } else {
#pragma unroll
    for (int bx = 0; bx < BOXES; ++bx) tma_load_2d(dst + bx * 2048, map, bx * BOX_ELEMS, row, bar, policy);
  }
}

// Byte offset of 16-byte chunk `chunk` (0 .. ROW_BYTES/16) of row `row` in a tile stored as
// 128-byte-swizzled boxes of 16 rows (box b at b*2048).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Two one-byte codes (the low 16 bits) of a narrow cache -> two f16 values, exactly.
template <typename KV>
__device__ __forceinline__ uint32_t widen2(uint32_t two_codes) {
  if constexpr (KV::code == PKV_INT8)
    return int8x2_to_f16x2(two_codes & 0xffffu);
  else
    return e4m3x2_to_f16x2(two_codes);
}

// Four one-byte codes -> two f16x2 words, exactly: lo = codes 0, 1 and hi = codes 2, 3. E4M3:
// the word's two 16-bit halves go straight to cvt.rn.f16x2.e4m3x2.
template <typename KV>
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (KV::code == PKV_INT8) {  // code + 128 under the exponent of 1024, minus 1152
    const uint32_t x = w ^ 0x80808080u;
    const __half2 bias = __half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
    uint32_t u = __byte_perm(x, 0x6464u, 0x5140u);
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&u), bias);
    lo = *reinterpret_cast<const uint32_t*>(&h);
    u = __byte_perm(x, 0x6464u, 0x5342u);
    h = __hsub2(*reinterpret_cast<const __half2*>(&u), bias);
    hi = *reinterpret_cast<const uint32_t*>(&h);
  } else {
    asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %2;\ncvt.rn.f16x2.e4m3x2 %0, a;\n"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  }
}

// K codes for the scores: as widen4, except that an INT8 code comes out as code + 1152 (the
// subtraction is left out). Every score of a (request, query head) then carries the same
// extra term 1152 * k_scale * sum(q), which the softmax cancels (a common shift of one row's
// scores; every chunk of the row gets the same one, so the split merge cancels it too). The
// biased values 1025..1279 are exact in f16 and the fp32 products and sums add only rounding.
template <typename KV>
__device__ __forceinline__ void widen4_scores(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (KV::code == PKV_INT8) {
    const uint32_t x = w ^ 0x80808080u;
    lo = __byte_perm(x, 0x6464u, 0x5140u);
    hi = __byte_perm(x, 0x6464u, 0x5342u);
  } else {
    widen4<KV>(w, lo, hi);
  }
}

// ---- pieces shared by the chunked and the balanced tensor-core decodes ---------------------

// Query fragments (MMA B operand of S^T = K Q^T), k order permuted as described above:
// lane (gid, tig) holds Q[g = 8 nt + gid][32 kp + 8 tig + 0..7] for every kp (bf16 path) or
// Q[g][16 (4 h + tig) + 0..15] for h = 0, 1 (FP8 path), read with 16-byte loads.
// FP8 / INT8 path: the MMAs take f16, whose range (max 65504, normal from 2^-14) is far
// narrower than bf16's or fp32's. Each query row is therefore multiplied by a power of two
// 2^e_g that puts its largest |q| in [2^14, 2^15) -- exact, so a bf16 q loses nothing -- and
// 2^-e_g goes into that head's score factor. An fp32 q is split into two f16 parts
// hi + lo (lo = the f16 rounding of q - hi), each contracted with K: 22 significant bits.
template <typename KV, typename TQ, int D, int G>
struct MmaQuery {
  static constexpr bool F8 = KV::bytes == 1;
  static constexpr bool QLO = F8 && sizeof(TQ) == 4;
  static constexpr int NT = (G + 7) / 8, KP = D / 32;
  uint32_t qf[NT][KP][4];
  uint32_t qlo[QLO ? NT : 1][QLO ? KP : 1][4];
  float sc_h[NT][2];  // score factor of heads 8 nt + 2 tig and 8 nt + 2 tig + 1 (log2 units)
};

// The query fragments of request b, KV head j.
template <typename KV, typename TQ, int D, int G>
__device__ __forceinline__ void mma_load_query(const DecodeArgs& a, int b, int j, int lane,
                                               MmaQuery<KV, TQ, D, G>& Q) {
  using QT = MmaQuery<KV, TQ, D, G>;
  constexpr bool F8 = QT::F8, QLO = QT::QLO;
  constexpr int NT = QT::NT, KP = QT::KP;
  const int gid = lane >> 2, tig = lane & 3;
  auto& qf = Q.qf;
  auto& qlo = Q.qlo;
  auto& sc_h = Q.sc_h;
  const float sc = a.scale_log2 * (F8 ? a.k_scales[j] : 1.f);
  {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int g = nt * 8 + gid;
      const bool live = g < G;
      const TQ* qrow = static_cast<const TQ*>(a.q) + ((size_t)b * a.h_q + j * G + (live ? g : 0)) * D;
      if constexpr (!F8) {
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (live) v = *reinterpret_cast<const uint4*>(qrow + 32 * kp + 8 * tig);
          qf[nt][kp][0] = v.x;
          qf[nt][kp][1] = v.y;
          qf[nt][kp][2] = v.z;
          qf[nt][kp][3] = v.w;
        }
        sc_h[nt][0] = sc_h[nt][1] = sc;
      } else {
        float x[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const TQ* src = qrow + 16 * (4 * h + tig);
#pragma unroll
          for (int k = 0; k < 16; k += (int)(16 / sizeof(TQ))) {
            if constexpr (sizeof(TQ) == 4) {
              float4 f = live ? *reinterpret_cast<const float4*>(src + k) : make_float4(0, 0, 0, 0);
              x[h][k] = f.x;
              x[h][k + 1] = f.y;
              x[h][k + 2] = f.z;
              x[h][k + 3] = f.w;
            } else {
              uint4 u = live ? *reinterpret_cast<const uint4*>(src + k) : make_uint4(0, 0, 0, 0);
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                x[h][k + 2 * t] = bf16lo(w[t]);
                x[h][k + 2 * t + 1] = bf16hi(w[t]);
              }
            }
          }
        }
        // largest |q| of head g: this lane's 32 values, then the 4 lanes (tig) sharing g
        float mx = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(x[h][k]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const int ex = (__float_as_int(mx) >> 23) & 0xff;  // biased exponent of the maximum
        // mx * 2^e in [2^14, 2^15) for a normal mx: e = 14 - (ex - 127); none for 0, inf, NaN
        const int e = (mx > 0.f && ex < 255) ? min(126, max(-126, 141 - ex)) : 0;
        const float up = __int_as_float((127 + e) << 23);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 16; ++k) x[h][k] *= up;
        // chunk 4h+tig of a K row holds k-steps 4h .. 4h+3, four values each
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const int kp = 2 * h + (ks >> 1), half = ks & 1;
            const float* v = &x[h][4 * ks];
            qf[nt][kp][2 * half] = pack_f16(v[0], v[1]);
            qf[nt][kp][2 * half + 1] = pack_f16(v[2], v[3]);
            if constexpr (QLO) {
              const __half2 h01 = *reinterpret_cast<const __half2*>(&qf[nt][kp][2 * half]);
              const __half2 h23 = *reinterpret_cast<const __half2*>(&qf[nt][kp][2 * half + 1]);
              qlo[nt][kp][2 * half] = pack_f16(v[0] - __low2float(h01), v[1] - __high2float(h01));
              qlo[nt][kp][2 * half + 1] =
                  pack_f16(v[2] - __low2float(h23), v[3] - __high2float(h23));
            }
          }
        // this lane's scores belong to heads 8 nt + 2 tig (+1): their exponents come from the
        // lanes holding those query rows (gid = 2 tig, 2 tig + 1)
        const int e0 = __shfl_sync(0xffffffffu, e, (2 * tig) * 4);
        const int e1 = __shfl_sync(0xffffffffu, e, (2 * tig + 1) * 4);
        sc_h[nt][0] = sc * __int_as_float((127 - e0) << 23);
        sc_h[nt][1] = sc * __int_as_float((127 - e1) << 23);
      }
    }
  }
}

// A warp's running softmax state over the pages it has read: per head the maximum and sum
// (log2 domain) and the weighted values, in MMA accumulator fragments.
// INT8 caches: the weighted values are accumulated over the biased codes (code + 1152, see
// widen4_scores), and p16_run keeps the sum of the f16 P values the MMAs used, so that the
// bias comes off once at the end: acc - 1152 sum(P) (the P products and their fp32 sums are
// the same as with unbiased codes, up to the accumulation's rounding of the larger terms).
template <int D, int G>
struct MmaRun {
  static constexpr int NT = (G + 7) / 8, MT = D / 16;
  float m_run[NT][2], l_run[NT][2], p16_run[NT][2];
  float acc[MT][NT][4];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
      p16_run[nt][0] = p16_run[nt][1] = 0.f;
#pragma unroll
      for (int mi = 0; mi < MT; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][nt][e] = 0.f;
    }
  }
};

// One staged (page, KV head) tile -- K at kt, V at vt (shared-memory addresses), logical page lp
// of a request of ctx tokens, nvalid rows before the context end -- folded into the warp's
// running state: scores, online softmax, weighted values.
template <typename KV, typename TQ, int D, int G>
__device__ __forceinline__ void mma_attend_page(uint32_t kt, uint32_t vt, int lp, int nvalid,
                                                int ctx, int sink, int window,
                                                const MmaQuery<KV, TQ, D, G>& Q,
                                                MmaRun<D, G>& R, uint16_t* pt, uint32_t pt_u32,
                                                int lane) {
  using QT = MmaQuery<KV, TQ, D, G>;
  constexpr bool F8 = QT::F8, QLO = QT::QLO;
  constexpr bool I8 = KV::code == PKV_INT8;
  constexpr int NT = QT::NT, KP = QT::KP, MT = D / 16;
  const int gid = lane >> 2, tig = lane & 3;
  const auto& qf = Q.qf;
  const auto& qlo = Q.qlo;
  const auto& sc_h = Q.sc_h;
  auto& m_run = R.m_run;
  auto& l_run = R.l_run;
  auto& p16_run = R.p16_run;
  auto& acc = R.acc;
  // ---- scores S^T[16 tokens][8 heads per n-tile] ----
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
  if constexpr (!F8) {
#pragma unroll
    for (int kp = 0; kp < KP; ++kp) {
      const uint4 r0 = lds128(kt + swz(gid, 4 * kp + tig));
      const uint4 r8 = lds128(kt + swz(gid + 8, 4 * kp + tig));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816<false>(s[nt], r0.x, r8.x, r0.y, r8.y, qf[nt][kp][0], qf[nt][kp][1]);
        mma16816<false>(s[nt], r0.z, r8.z, r0.w, r8.w, qf[nt][kp][2], qf[nt][kp][3]);
      }
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // 16-byte chunk 4h+tig of a row = 4 k-steps x 4 codes
      const uint4 r0 = lds128(kt + swz(gid, 4 * h + tig));
      const uint4 r8 = lds128(kt + swz(gid + 8, 4 * h + tig));
      const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w};
      const uint32_t w8[4] = {r8.x, r8.y, r8.z, r8.w};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a0, a1, a2, a3;
        widen4_scores<KV>(w0[ks], a0, a2);
        widen4_scores<KV>(w8[ks], a1, a3);
        const int kp = 2 * h + (ks >> 1), half = ks & 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816<true>(s[nt], a0, a1, a2, a3, qf[nt][kp][2 * half],
                         qf[nt][kp][2 * half + 1]);
          if constexpr (QLO)
            mma16816<true>(s[nt], a0, a1, a2, a3, qlo[nt][kp][2 * half],
                           qlo[nt][kp][2 * half + 1]);
        }
      }
    }
  }

  // ---- online softmax: lane holds tokens gid, gid+8 of heads 8nt+2tig, 8nt+2tig+1 ----
  const bool v0 = attended(lp * kPageSize + gid, ctx, sink, window);
  const bool v8 = attended(lp * kPageSize + gid + 8, ctx, sink, window);
  float alpha[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] = v0 ? s[nt][0] * sc_h[nt][0] : -INFINITY;
    s[nt][1] = v0 ? s[nt][1] * sc_h[nt][1] : -INFINITY;
    s[nt][2] = v8 ? s[nt][2] * sc_h[nt][0] : -INFINITY;
    s[nt][3] = v8 ? s[nt][3] * sc_h[nt][1] : -INFINITY;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float mx = fmaxf(s[nt][k], s[nt][k + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[nt][k], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[nt][k] = exp2f(m_run[nt][k] - m_use);
      s[nt][k] = exp2f(s[nt][k] - m_use);
      s[nt][k + 2] = exp2f(s[nt][k + 2] - m_use);
      l_run[nt][k] = l_run[nt][k] * alpha[nt][k] + s[nt][k] + s[nt][k + 2];
      m_run[nt][k] = m_new;
    }
    // P^T into the warp buffer: pt[g][t], g = 8nt + 2tig (+1), t = gid (+8)
    uint16_t* row0 = pt + (nt * 8 + 2 * tig) * kPageSize;
    uint16_t* row1 = row0 + kPageSize;
    if constexpr (F8) {
      const __half h0 = __float2half_rn(s[nt][0]), h1 = __float2half_rn(s[nt][1]);
      const __half h2 = __float2half_rn(s[nt][2]), h3 = __float2half_rn(s[nt][3]);
      if constexpr (I8) {
        p16_run[nt][0] = p16_run[nt][0] * alpha[nt][0] + __half2float(h0) + __half2float(h2);
        p16_run[nt][1] = p16_run[nt][1] * alpha[nt][1] + __half2float(h1) + __half2float(h3);
      }
      row0[gid] = __half_as_ushort(h0);
      row1[gid] = __half_as_ushort(h1);
      row0[gid + 8] = __half_as_ushort(h2);
      row1[gid + 8] = __half_as_ushort(h3);
    } else {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(s[nt][0]);
      const __nv_bfloat16 h1 = __float2bfloat16_rn(s[nt][1]);
      const __nv_bfloat16 h2 = __float2bfloat16_rn(s[nt][2]);
      const __nv_bfloat16 h3 = __float2bfloat16_rn(s[nt][3]);
      row0[gid] = __bfloat16_as_ushort(h0);
      row1[gid] = __bfloat16_as_ushort(h1);
      row0[gid + 8] = __bfloat16_as_ushort(h2);
      row1[gid + 8] = __bfloat16_as_ushort(h3);
    }
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      acc[mi][nt][0] *= alpha[nt][0];
      acc[mi][nt][1] *= alpha[nt][1];
      acc[mi][nt][2] *= alpha[nt][0];
      acc[mi][nt][3] *= alpha[nt][1];
    }
  }

  // ---- O^T[dims][heads] += V^T P^T ----
  if constexpr (!F8) {
    if (nvalid < kPageSize) {
      // zero the stale rows of the last page (16 chunks of 16 bytes per row)
      for (int e = lane; e < (kPageSize - nvalid) * 16; e += 32) {
        const int r = nvalid + (e >> 4), ch = e & 15;
        sts128(vt + swz(r, ch), make_uint4(0, 0, 0, 0));
      }
    }
  }
  __syncwarp();
  uint32_t pb[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t rowg = pt_u32 + (nt * 8 + gid) * kPageSize * 2;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(pb[nt][0]) : "r"(rowg + 4 * tig));
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(pb[nt][1]) : "r"(rowg + 16 + 4 * tig));
  }
  if constexpr (!F8) {
    // V^T fragments straight from the swizzled bf16 tile: m-tile mi covers dims 16 mi ..
    const int q = lane >> 3, rr = lane & 7;
    const int t = (q >> 1) * 8 + rr;
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(vt + swz(t, 2 * mi + (q & 1)), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma16816<false>(acc[mi][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
    }
  } else {
    // V^T fragments built in registers from the FP8 tile. The lane reads 16 codes (dims
    // 16 gid .. 16 gid + 15) of tokens 2tig, 2tig+1, 2tig+8, 2tig+9; byte permutes pair
    // each dim's codes of consecutive tokens, which widen exactly to f16. Row gid of m-tile
    // mi is dim 16 gid + 2 mi and row gid + 8 is dim 16 gid + 2 mi + 1 (undone in the merge).
    uint4 vr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = 2 * tig + (k & 1) + 8 * (k >> 1);
      vr[k] = lds128(vt + swz(r, gid));
      if (r >= nvalid) vr[k] = make_uint4(0, 0, 0, 0);  // stale rows of the last page
    }
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      const int wi = mi >> 1;
      const uint32_t sel = (mi & 1) ? 0x7362u : 0x5140u;
      const uint32_t w0 = wi == 0 ? vr[0].x : wi == 1 ? vr[0].y : wi == 2 ? vr[0].z : vr[0].w;
      const uint32_t w1 = wi == 0 ? vr[1].x : wi == 1 ? vr[1].y : wi == 2 ? vr[1].z : vr[1].w;
      const uint32_t w2 = wi == 0 ? vr[2].x : wi == 1 ? vr[2].y : wi == 2 ? vr[2].z : vr[2].w;
      const uint32_t w3 = wi == 0 ? vr[3].x : wi == 1 ? vr[3].y : wi == 2 ? vr[3].z : vr[3].w;
      const uint32_t lo = __byte_perm(w0, w1, sel);  // tokens 2tig, 2tig+1
      const uint32_t hi = __byte_perm(w2, w3, sel);  // tokens 2tig+8, 2tig+9
      uint32_t a0, a1, a2, a3;
      widen4_scores<KV>(lo, a0, a1);  // (INT8: biased codes; the bias comes off at the end)
      widen4_scores<KV>(hi, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma16816<true>(acc[mi][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
    }
  }
}

// A warp's state into its merge area: [G][D] weighted values, [G] maxima, [G] sums.
template <typename KV, int D, int G>
__device__ __forceinline__ void mma_run_to_smem(const MmaRun<D, G>& R, float* red_acc,
                                                float* red_m, float* red_l, int lane) {
  constexpr bool F8 = KV::bytes == 1;
  constexpr bool I8 = KV::code == PKV_INT8;
  constexpr int NT = MmaRun<D, G>::NT, MT = MmaRun<D, G>::MT;
  const int gid = lane >> 2, tig = lane & 3;
  const auto& m_run = R.m_run;
  const auto& l_run = R.l_run;
  const auto& acc = R.acc;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float l = l_run[nt][k];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int g = nt * 8 + 2 * tig + k;
      if (gid == 0 && g < G) {
        red_m[g] = m_run[nt][k];
        red_l[g] = l;
      }
      float bias = 0.f;  // INT8: 1152 times the head's sum of the P values the MMAs used
      if constexpr (I8) {
        float p = R.p16_run[nt][k];
        p += __shfl_xor_sync(0xffffffffu, p, 4);
        p += __shfl_xor_sync(0xffffffffu, p, 8);
        p += __shfl_xor_sync(0xffffffffu, p, 16);
        bias = 1152.f * p;
      }
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) {
        if (g < G) {
          // dims of rows gid and gid+8 of m-tile mi (see the two V^T fragment layouts)
          const int i0 = F8 ? 16 * gid + 2 * mi : 16 * mi + gid;
          const int i1 = F8 ? i0 + 1 : i0 + 8;
          red_acc[g * D + i0] = acc[mi][nt][k] - bias;
          red_acc[g * D + i1] = acc[mi][nt][k + 2] - bias;
        }
      }
    }
  }
}

// WU (warp per request): every request has a single chunk; warp w of CTA z takes request
// NW z + w whole (its pages 0, 1, 2, ... through its own two ring stages) and writes its output
// itself; the warps of a CTA only share the barrier set-up.
template <typename KV, typename TQ, int D, int G, bool WU>
__global__ void __launch_bounds__(32 * PKV_MMA_WARPS) paged_decode_mma_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using S = MmaShape<KV, D, G, WU>;
  constexpr bool F8 = S::kFp8;
  constexpr int NW = S::kWarps, SPW = S::SPW, NT = S::NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, j = blockIdx.y;
  const bool warp_live = !WU || (int)blockIdx.z * NW + warp < a.batch;
  const int b = WU ? (warp_live ? (int)blockIdx.z * NW + warp : 0) : (int)blockIdx.z;
  const bool reporter = c == 0 && (WU ? lane == 0 && warp_live : threadIdx.x == 0);
  int ctx = max(0, a.context_lens[b]);
  const bool cut = ctx > a.max_pages * kPageSize;
  if (cut) {  // longer than its page table: read what the table holds, append nothing
    if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
    ctx = a.max_pages * kPageSize;
  }
  const SeqPlan plan = seq_plan(a, b, ctx);
  if (plan.prefix > 0 && ctx < plan.prefix * kPageSize + (a.k_new != nullptr ? 1 : 0)) {
    // a cascade member's context must reach past its group's shared pages
    if (reporter) atomicOr(a.err, PKV_DEVERR_BAD_GROUP);
  }
  const SeqPages sp = plan.sp;
  const int pages_seq = sp.n;  // the pages read here, split into n_chunks near-equal chunks
  const int n_chunks = plan.n_chunks;
  // the combine kernel (a programmatic dependent launch) may be scheduled once every CTA of
  // this grid has started; it waits for this grid's completion before reading its partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!WU && c > 0 && c >= n_chunks) return;
  const bool active = warp_live && !(c > 0 && c >= n_chunks);  // (WU: per warp)
  const int per_chunk = n_chunks > 0 ? (pages_seq + n_chunks - 1) / n_chunks : 0;
  const int page0 = c * per_chunk;
  const int n_pages = active ? max(0, min(per_chunk, pages_seq - page0)) : 0;
  // the warp that will reach the page of position ctx-1 prefetches this step's rows now
  const int append_warp =
      active && a.k_new != nullptr && !cut && n_pages > 0 && page0 + n_pages == pages_seq
          ? (WU ? warp : (n_pages - 1) % PKV_MMA_WARPS)
          : -1;
  if (warp == append_warp) append_prefetch<KV, D>(a, b, j, lane);
  // (as a dependent launch of the prefix kernel, its partials are not written yet)
  if (active && plan.slot0 > 0 && n_chunks <= 1 && !a.prefix_dep) {
    if constexpr (WU)
      prefetch_prefix_partials<D, G, 32>(a, b, j, plan.slot0, lane);
    else
      prefetch_prefix_partials<D, G, 32 * PKV_MMA_WARPS>(a, b, j, plan.slot0, threadIdx.x);
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + S::BIG_BYTES) + warp * NT * 8 * kPageSize;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BIG_BYTES + S::PT_BYTES);
  int* page_ok = reinterpret_cast<int*>(full + S::STAGES);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  __syncthreads();
  if (WU && !active) return;  // (no CTA-wide barrier follows in this mode)

  const int32_t* btrow = a.block_tables + (size_t)b * a.max_pages;
  const uint64_t pol = l2_evict_first_policy();
  const uint32_t ring_u32 = smem_u32(ring);

  auto issue = [&](int i, int stg, int pid) {  // lane 0: page i of the chunk (id pid) -> stage stg
    if (pid < 0 || pid >= a.num_pages) {
      page_ok[stg] = 0;
      atomicOr(a.err, PKV_DEVERR_BAD_PAGE);
      mbar_arrive(&full[stg]);
    } else {
      page_ok[stg] = 1;
      mbar_arrive_expect_tx(&full[stg], S::STAGE_BYTES);
      const int row = (pid * a.h_kv + j) * kPageSize;
      const uint32_t dst = ring_u32 + stg * S::STAGE_BYTES;
      tma_tile<S::BOXES, S::BOX_ELEMS>(dst, &tm_k, a.tma_rank, row, &full[stg], pol);
      tma_tile<S::BOXES, S::BOX_ELEMS>(dst + S::TILE_BYTES, &tm_v, a.tma_rank, row, &full[stg],
                                       pol);
    }
  };

  // the warp's pages: chunk pages w, w + NW, ... (WU: all of them)
  constexpr int STRIDE = WU ? 1 : NW;
  const int first = WU ? 0 : warp;
  const int n_mine = WU ? n_pages : (n_pages > warp ? (n_pages - warp + NW - 1) / NW : 0);
  // Page ids of the warp's pages, read 32 at a time ahead of their copies so that no copy waits
  // on a table read: lane L holds the id of the warp's page 32 t + L.
  int ids = -1;
  auto load_ids = [&](int t) {
    const int mm = 32 * t + lane;
    ids = mm < n_mine ? btrow[logical_page(sp, page0 + first + STRIDE * mm)] : -1;
  };
  load_ids(0);
  {
    int first_ids[SPW];
#pragma unroll
    for (int m = 0; m < SPW; ++m) first_ids[m] = __shfl_sync(0xffffffffu, ids, m);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < SPW; ++m)
        if (m < n_mine) issue(first + STRIDE * m, warp * SPW + m, first_ids[m]);
    }
  }

  MmaQuery<KV, TQ, D, G> Q;
  mma_load_query<KV, TQ, D, G>(a, b, j, lane, Q);

  MmaRun<D, G> R;
  R.reset();
  const uint32_t pt_u32 = smem_u32(pt);

  int m = 0;
  bool ok = true;
  for (; m < n_mine; ++m) {
    const int i = first + STRIDE * m;
    const int stg = warp * SPW + (m % SPW);
    const bool got = mbar_wait(&full[stg], (m / SPW) & 1, a.err);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    if (page_ok[stg]) {
      const int lp = logical_page(sp, page0 + i);
      const int nvalid = min(kPageSize, ctx - lp * kPageSize);  // rows before the context end
      const uint32_t kt = ring_u32 + stg * S::STAGE_BYTES;
      const uint32_t vt = kt + S::TILE_BYTES;
      if (warp == append_warp && i == n_pages - 1) {
        uint8_t* ktp = ring + stg * S::STAGE_BYTES;
        fused_append_row<KV, D>(a, b, j, btrow[lp], nvalid - 1, ktp, ktp + S::TILE_BYTES, lane,
                                [](int r, int ch) { return (int)swz(r, ch); });
        __syncwarp();
      }

      mma_attend_page<KV, TQ, D, G>(kt, vt, lp, nvalid, ctx, a.sink, a.window, Q, R, pt, pt_u32,
                                    lane);
    }
    __syncwarp();
    if (m + SPW < n_mine) {  // warp-uniform
      const int mn = m + SPW;
      if ((mn & 31) == 0) load_ids(mn >> 5);
      const int pid = __shfl_sync(0xffffffffu, ids, mn & 31);
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(i + STRIDE * SPW, stg, pid);
      }
    }
  }
  if (!ok && lane == 0) {
    for (int mm = m; mm < n_mine && mm < m + SPW; ++mm)
      mbar_wait(&full[warp * SPW + (mm % SPW)], (mm / SPW) & 1, a.err);
  }
  if constexpr (WU)
    __syncwarp();
  else
    __syncthreads();  // every copy has landed: the ring is free for the merge

  // the merge area: [NW][G][D] values, [NW][G] maxima, [NW][G] sums (WU: past the ring)
  float* red_acc = reinterpret_cast<float*>(ring + (WU ? S::RING_BYTES : 0));
  float* red_m = red_acc + NW * G * D;
  float* red_l = red_m + NW * G;
  mma_run_to_smem<KV, D, G>(R, red_acc + warp * G * D, red_m + warp * G, red_l + warp * G, lane);
  const float vs = F8 ? a.v_scales[j] : 1.f;
  // a dependent launch of the prefix kernel: its partials are complete and visible past here
  if (a.prefix_dep && !a.defer_fold) asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (WU) {
    __syncwarp();
    decode_epilogue_warp<TQ, D, G>(a, b, j, plan.slot0, red_acc + warp * G * D, red_m + warp * G,
                                   red_l + warp * G, vs, lane);
  } else {
    __syncthreads();
    decode_epilogue<TQ, D, G, NW, S::kThreads>(a, b, j, c, n_chunks, plan.slot0, red_acc,
                                               red_m, red_l, vs);
  }
  // deferred fold: the combine waits for this grid only, so this grid must not complete before
  // the prefix kernel; one thread of the first CTA (always active) waits for it, at its end
  if (a.defer_fold && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename KV, typename TQ, int D, int G, bool WU>
cudaError_t launch_decode_mma_w(const DecodeArgs& a, const CUtensorMap& tk,
                                const CUtensorMap& tv, cudaStream_t s) {
  using S = MmaShape<KV, D, G, WU>;
  auto kern = paged_decode_mma_kernel<KV, TQ, D, G, WU>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device, per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_done.load() >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done.fetch_or(1ull << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.chunk_grid, a.h_kv, WU ? (a.batch + S::kWarps - 1) / S::kWarps : a.batch);
  cfg.blockDim = dim3(S::kThreads);
  cfg.dynamicSmemBytes = S::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.prefix_dep ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, tk, tv);
}

template <typename KV, typename TQ, int D, int G>
cudaError_t launch_decode_mma_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s) {
  return a.warp_units ? launch_decode_mma_w<KV, TQ, D, G, true>(a, tk, tv, s)
                      : launch_decode_mma_w<KV, TQ, D, G, false>(a, tk, tv, s);
}

template <typename KV, typename TQ>
cudaError_t launch_decode_mma_g(const DecodeArgs& a, int group, const CUtensorMap& tk,
                                const CUtensorMap& tv, cudaStream_t s) {
  switch (group) {
    case 1: return launch_decode_mma_t<KV, TQ, 128, 1>(a, tk, tv, s);
    case 2: return launch_decode_mma_t<KV, TQ, 128, 2>(a, tk, tv, s);
    case 4: return launch_decode_mma_t<KV, TQ, 128, 4>(a, tk, tv, s);
    case 8: return launch_decode_mma_t<KV, TQ, 128, 8>(a, tk, tv, s);
    case 16: return launch_decode_mma_t<KV, TQ, 128, 16>(a, tk, tv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
