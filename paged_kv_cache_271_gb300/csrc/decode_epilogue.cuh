// End of a decode CTA, shared by the CUDA-core and tensor-core kernels: the CTA's warps have
// left their (running max, sum, weighted values) per head in shared memory; merge them, then
//  * the request's only chunk: write out = acc / l -- in a cascade decode that folds in the
//    decode kernel, after merging in the partials of the request's shared prefix (chunk slots
//    0 .. slot0 - 1, written by the prefix kernel);
//  * one of several chunks, or a cascade member's chunk when the combine kernel folds: write
//    this chunk's partial (m, l, acc) to chunk slot slot0 + c;
//    when the call merges in place, the last CTA of the (request, KV head) to finish -- found
//    with a counter in the workspace -- merges every slot of the group in slot order and
//    writes out, then resets the counter to 0 for the next call. Otherwise a separate combine
//    kernel merges the partials.
#pragma once

#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <typename TQ, int D, int G, int NW, int NTHR>
__device__ __forceinline__ void decode_epilogue(const DecodeArgs& a, int b, int j, int c,
                                                int n_chunks, int slot0, const float* red_acc,
                                                const float* red_m, const float* red_l,
                                                float vs) {
  __shared__ int s_last;
  // this CTA finishes the request (with a deferred fold, a cascade member's prefix partials
  // are merged by the combine kernel instead)
  const bool direct = n_chunks <= 1 && !(a.defer_fold && slot0 > 0);
  for (int e = threadIdx.x; e < G * D; e += NTHR) {
    const int g = e / D, i = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * G + g]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float wt = exp2f(red_m[w * G + g] - M);
        L = fmaf(wt, red_l[w * G + g], L);
        A = fmaf(wt, red_acc[(w * G + g) * D + i], A);
      }
    }
    A *= vs;
    const size_t bh = (size_t)b * a.h_q + j * G + g;
    if (direct) {
      if (slot0 > 0) {  // fold in the shared prefix's partials, 8 slots per batch of loads
        const float* ml = a.ws_ml + bh * a.n_chunk_slots * 2;
        const float* acc = a.ws_acc + bh * a.n_chunk_slots * D + i;
        for (int k0 = 0; k0 < slot0; k0 += 8) {
          float mv[8], lv[8], av[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const bool in = k0 + u < slot0;
            mv[u] = in ? ml[2 * (k0 + u)] : -INFINITY;
            lv[u] = in ? ml[2 * (k0 + u) + 1] : 0.f;
            av[u] = in ? acc[(size_t)(k0 + u) * D] : 0.f;
          }
          float Mb = M;
#pragma unroll
          for (int u = 0; u < 8; ++u) Mb = fmaxf(Mb, mv[u]);
          if (Mb == -INFINITY) continue;
          const float w0 = exp2f(M - Mb);
          L *= w0;
          A *= w0;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float w = exp2f(mv[u] - Mb);
            L = fmaf(w, lv[u], L);
            A = fmaf(w, av[u], A);
          }
          M = Mb;
        }
      }
      store_from_float(static_cast<TQ*>(a.out), bh * D + i, L > 0.f ? A / L : 0.f);
    } else {
      const size_t part = bh * a.n_chunk_slots + slot0 + c;
      a.ws_acc[part * D + i] = A;
      if (i == 0) {
        a.ws_ml[part * 2 + 0] = M;
        a.ws_ml[part * 2 + 1] = L;
      }
    }
  }
  if (direct || !a.merge_in_place) return;

  // Publish this chunk's partial, then count it: after the barrier one thread's fence orders
  // the whole CTA's partial before the count (fences are cumulative), and the CTA that brings
  // the count to n_chunks fences again before reading the other chunks' partials from L2.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(a.counters + (size_t)b * a.h_kv + j, 1);
    s_last = (prev == n_chunks - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  const int n_total = slot0 + n_chunks;
  for (int e = threadIdx.x; e < G * D; e += NTHR) {
    const int g = e / D, i = e % D;
    const size_t bh = (size_t)b * a.h_q + j * G + g;
    const float* ml = a.ws_ml + bh * a.n_chunk_slots * 2;
    const float* acc = a.ws_acc + bh * a.n_chunk_slots * D + i;
    float M = -INFINITY;
    for (int k = 0; k < n_total; ++k) M = fmaxf(M, __ldcg(ml + 2 * k));
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int k = 0; k < n_total; ++k) {
        const float w = exp2f(__ldcg(ml + 2 * k) - M);
        L = fmaf(w, __ldcg(ml + 2 * k + 1), L);
        A = fmaf(w, __ldcg(acc + (size_t)k * D), A);
      }
    }
    store_from_float(static_cast<TQ*>(a.out), bh * D + i, L > 0.f ? A / L : 0.f);
  }
  if (threadIdx.x == 0) a.counters[(size_t)b * a.h_kv + j] = 0;
}

// The same for one warp that owns a whole (request, KV head) run of a launch in which every
// request has a single chunk (warp-per-request decode): the warp's merged values are in its own
// [G][D] area. Lane L owns dims 4L .. 4L+3 (D = 128) of every head, so a cascade member's prefix
// partials come in with one 16-byte load per (head, slot), all heads' loads at once.
template <typename TQ, int D, int G>
__device__ __forceinline__ void decode_epilogue_warp(const DecodeArgs& a, int b, int j,
                                                     int slot0, const float* red_acc,
                                                     const float* red_m, const float* red_l,
                                                     float vs, int lane) {
  static_assert(D == 128, "four dims per lane");
  const int i0 = 4 * lane;
  float M[G], L[G], A[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = red_m[g];
    L[g] = M[g] != -INFINITY ? red_l[g] : 0.f;
    const float4 v = *reinterpret_cast<const float4*>(red_acc + g * D + i0);
    const bool live = M[g] != -INFINITY;
    A[g][0] = live ? v.x * vs : 0.f;
    A[g][1] = live ? v.y * vs : 0.f;
    A[g][2] = live ? v.z * vs : 0.f;
    A[g][3] = live ? v.w * vs : 0.f;
  }
  if (a.defer_fold && slot0 > 0) {  // the own pages' partial, at slot slot0 (the combine merges)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const size_t part = ((size_t)b * a.h_q + j * G + g) * a.n_chunk_slots + slot0;
      *reinterpret_cast<float4*>(a.ws_acc + part * D + i0) =
          make_float4(A[g][0], A[g][1], A[g][2], A[g][3]);
      if (lane == 0) {
        a.ws_ml[part * 2] = M[g];
        a.ws_ml[part * 2 + 1] = L[g];
      }
    }
    return;
  }
  constexpr int KB = G <= 4 ? 4 : (G <= 8 ? 2 : 1);  // slots whose loads go out together
  for (int k0 = 0; k0 < slot0; k0 += KB) {  // fold in the prefix partials
    float mv[KB][G], lv[KB][G];
    float4 av[KB][G];
#pragma unroll
    for (int u = 0; u < KB; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const bool in = k0 + u < slot0;
        const size_t part =
            ((size_t)b * a.h_q + j * G + g) * a.n_chunk_slots + (in ? k0 + u : 0);
        mv[u][g] = in ? a.ws_ml[part * 2] : -INFINITY;
        lv[u][g] = in ? a.ws_ml[part * 2 + 1] : 0.f;
        av[u][g] = in ? *reinterpret_cast<const float4*>(a.ws_acc + part * D + i0)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int u = 0; u < KB; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float Mb = fmaxf(M[g], mv[u][g]);
        if (Mb == -INFINITY) continue;
        const float w0 = exp2f(M[g] - Mb), w = exp2f(mv[u][g] - Mb);
        L[g] = fmaf(w, lv[u][g], L[g] * w0);
        A[g][0] = fmaf(w, av[u][g].x, A[g][0] * w0);
        A[g][1] = fmaf(w, av[u][g].y, A[g][1] * w0);
        A[g][2] = fmaf(w, av[u][g].z, A[g][2] * w0);
        A[g][3] = fmaf(w, av[u][g].w, A[g][3] * w0);
        M[g] = Mb;
      }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const size_t o = ((size_t)b * a.h_q + j * G + g) * D + i0;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      store_from_float(static_cast<TQ*>(a.out), o + t, L[g] > 0.f ? A[g][t] / L[g] : 0.f);
  }
}

}  // namespace pkv

namespace pkv {

// Decode step with the append fused in: the CTA that reads the page holding position ctx-1 of
// request b (KV head j) writes this step's K and V rows there -- into the pools and into its
// shared-memory copy of the page -- before using the page. Same bytes as kv_append: a copy
// for bf16/fp32 caches, cvt.rn.satfinite.e4m3(fp32(x / s)) for FP8, the clamped nearest-even
// integer of fp32(x / s) for INT8.
//
// The appending warp prefetches its share of the new rows into L1 as soon as the kernel starts
// (append_prefetch), so that the reads at the page hit.
template <typename KV, int D>
struct AppendRow {
  static constexpr int NCH = D * KV::bytes / 16;  // 16-byte chunks per output row
  static constexpr int PER = (2 * NCH + 31) / 32;  // chunks per lane
  uint4 raw[PER][4];  // the chunk's inputs: up to 16 fp32 values
};

template <typename KV, int D>
__device__ __forceinline__ void append_prefetch(const DecodeArgs& a, int b, int j, int lane) {
  const int in_bytes = a.new_dtype == PKV_F32 ? 4 : 2;
  const int row = D * in_bytes;  // bytes of one new row (K or V)
  const size_t off = ((size_t)b * a.h_kv + j) * row;
  for (int e = lane; e < 2 * row / 128; e += 32) {
    const char* base = static_cast<const char*>(e < row / 128 ? a.k_new : a.v_new);
    asm volatile("prefetch.global.L1 [%0];" ::"l"(base + off + 128 * (e % (row / 128))));
  }
}

template <typename KV, int D>
__device__ __forceinline__ void append_load(const DecodeArgs& a, int b, int j, int lane,
                                            AppendRow<KV, D>& ar) {
  constexpr int NCH = AppendRow<KV, D>::NCH;
  const size_t src_elem = ((size_t)b * a.h_kv + j) * D;
#pragma unroll
  for (int k = 0; k < AppendRow<KV, D>::PER; ++k) {
    const int e = lane + 32 * k;
    if (e >= 2 * NCH) continue;
    const bool isv = e >= NCH;
    const int ch = isv ? e - NCH : e;
    const void* src = isv ? a.v_new : a.k_new;
    if constexpr (KV::bytes == 1) {
      const int n16 = a.new_dtype == PKV_BF16 ? 2 : 4;  // 16 inputs in 2 or 4 vectors
      const uint4* p = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(src) + (src_elem + 16 * ch) * (n16 == 2 ? 2 : 4));
#pragma unroll
      for (int h = 0; h < 4; ++h) ar.raw[k][h] = h < n16 ? p[h] : make_uint4(0, 0, 0, 0);
    } else {
      ar.raw[k][0] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(src) +
                                                      src_elem * KV::bytes + 16 * ch);
    }
  }
}

// off(r, ch) is the byte offset of 16-byte chunk ch of row r in a shared-memory tile.
template <typename KV, int D, typename OffFn>
__device__ __forceinline__ void append_store(const DecodeArgs& a, int j, int pid, int r,
                                             uint8_t* k_tile, uint8_t* v_tile, int lane,
                                             OffFn off, const AppendRow<KV, D>& ar) {
  constexpr int NCH = AppendRow<KV, D>::NCH;
  const size_t row_byte = ((((size_t)pid * a.h_kv + j) * kPageSize + r) * D) * KV::bytes;
#pragma unroll
  for (int k = 0; k < AppendRow<KV, D>::PER; ++k) {
    const int e = lane + 32 * k;
    if (e >= 2 * NCH) continue;
    const bool isv = e >= NCH;
    const int ch = isv ? e - NCH : e;
    uint4 val;
    if constexpr (KV::bytes == 1) {
      float x[16];
      if (a.new_dtype == PKV_BF16) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w[4] = {ar.raw[k][h].x, ar.raw[k][h].y, ar.raw[k][h].z, ar.raw[k][h].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            x[8 * h + 2 * t] = bf16lo(w[t]);
            x[8 * h + 2 * t + 1] = bf16hi(w[t]);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          x[4 * h] = __uint_as_float(ar.raw[k][h].x);
          x[4 * h + 1] = __uint_as_float(ar.raw[k][h].y);
          x[4 * h + 2] = __uint_as_float(ar.raw[k][h].z);
          x[4 * h + 3] = __uint_as_float(ar.raw[k][h].w);
        }
      }
      const float s = isv ? a.v_scales[j] : a.k_scales[j];
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (KV::code == PKV_INT8) {
          uint32_t acc = 0;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = min(127, max(-127, __float2int_rn(__fdiv_rn(x[4 * q + t], s))));
            acc |= ((uint32_t)(c & 0xff)) << (8 * t);
          }
          w[q] = acc;
        } else {
          const uint16_t lo = static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[4 * q], s), __fdiv_rn(x[4 * q + 1], s)), __NV_SATFINITE,
              __NV_E4M3));
          const uint16_t hi = static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[4 * q + 2], s), __fdiv_rn(x[4 * q + 3], s)),
              __NV_SATFINITE, __NV_E4M3));
          w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
      }
      val = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      val = ar.raw[k][0];
    }
    *reinterpret_cast<uint4*>((isv ? v_tile : k_tile) + off(r, ch)) = val;
    uint8_t* pool = static_cast<uint8_t*>(const_cast<void*>(isv ? a.v_cache : a.k_cache));
    *reinterpret_cast<uint4*>(pool + row_byte + 16 * ch) = val;
  }
}

// Both steps at once (for callers that do not read ahead).
template <typename KV, int D, typename OffFn>
__device__ __forceinline__ void fused_append_row(const DecodeArgs& a, int b, int j, int pid,
                                                 int r, uint8_t* k_tile, uint8_t* v_tile,
                                                 int lane, OffFn off) {
  AppendRow<KV, D> ar;
  append_load<KV, D>(a, b, j, lane, ar);
  append_store<KV, D>(a, j, pid, r, k_tile, v_tile, lane, off, ar);
}

// The partials of a cascade member's shared prefix that the epilogue will fold in: prefetched
// into L1 when the CTA starts, one 128-byte line per thread.
template <int D, int G, int NTHR>
__device__ __forceinline__ void prefetch_prefix_partials(const DecodeArgs& a, int b, int j,
                                                         int slot0, int tid) {
  const int lines = slot0 * D * 4 / 128 + 2;  // weighted values, then the (max, sum) pairs
  for (int e = tid; e < G * lines; e += NTHR) {
    const int g = e / lines, k = e % lines;
    const size_t bh = (size_t)b * a.h_q + j * G + g;
    const char* p =
        k < lines - 2 ? reinterpret_cast<const char*>(a.ws_acc + bh * a.n_chunk_slots * D) + 128 * k
                      : reinterpret_cast<const char*>(a.ws_ml + bh * a.n_chunk_slots * 2) +
                            (k == lines - 1 ? 8 * slot0 - 4 : 0);
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
  }
}

}  // namespace pkv
