// Device-side helpers shared by the library's kernels: element conversions, shared-memory
// barriers (mbarrier) with bounded waits, and 1-D bulk copies global -> shared.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPageSize = 16;
// A bounded wait gives up after this long; the kernel then records PKV_DEVERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Storage tags for the three cache element types.
struct F32 {
  using storage = float;
  static constexpr int bytes = 4;
  static constexpr int code = PKV_F32;
};
struct BF16 {
  using storage = __nv_bfloat16;
  static constexpr int bytes = 2;
  static constexpr int code = PKV_BF16;
};
struct FP8 {
  using storage = uint8_t;
  static constexpr int bytes = 1;
  static constexpr int code = PKV_FP8_E4M3;
};
struct INT8 {
  using storage = int8_t;
  static constexpr int bytes = 1;
  static constexpr int code = PKV_INT8;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- which pages a request attends ----------------------------------------------------------

// With a sliding window of W positions (plus S attention sinks) a request of ctx tokens attends
// positions t >= ctx - W and t < S; without a window (W = 0) every position. Its attended
// pages, in logical order, are numbered 0 .. n-1: the first `sink_pages` are logical pages
// 0 .. sink_pages-1, the rest logical pages win_first, win_first + 1, ... Pages holding no
// attended position are not read (their table entries may be released).
struct SeqPages {
  int n;
  int sink_pages;
  int win_first;
};

__device__ __forceinline__ SeqPages seq_pages(int ctx, int sink, int window) {
  const int pages = (ctx + kPageSize - 1) / kPageSize;
  SeqPages r{pages, pages, pages};
  if (window > 0) {
    const int wp = max(0, ctx - window) / kPageSize;
    const int sp = min((max(0, sink) + kPageSize - 1) / kPageSize, pages);
    if (wp > sp) r = SeqPages{sp + (pages - wp), sp, wp};
  }
  return r;
}

__device__ __forceinline__ int logical_page(const SeqPages& s, int v) {
  return v < s.sink_pages ? v : s.win_first + (v - s.sink_pages);
}

__device__ __forceinline__ bool attended(int t, int ctx, int sink, int window) {
  return t < ctx && (window <= 0 || t >= ctx - window || t < sink);
}

// ---- mbarrier ------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete. Gives up after kWaitLimitNs, sets
// PKV_DEVERR_TIMEOUT in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, PKV_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---- bulk copies (TMA, untiled) -----------------------------------------------------------

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing as transaction bytes on `bar`. The source is streamed (L2 evict-first).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---- element conversions (all exact) -------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two E4M3 codes (low byte first) -> two floats, via the exact e4m3 -> f16 conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  return __half22float2(__half2(h));
}

// Two INT8 codes (low byte first) -> two f16 (exact): biasing the byte by 128 and placing it
// under the f16 exponent of 1024 gives 1024 + (c + 128); subtracting 1152 leaves c.
__device__ __forceinline__ uint32_t int8x2_to_f16x2(uint32_t two_codes) {
  const uint32_t u = __byte_perm(two_codes ^ 0x8080u, 0x6464u, 0x5140u);
  __half2 h = *reinterpret_cast<const __half2*>(&u);
  h = __hsub2(h, __half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u)));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Loads DL consecutive elements of a shared-memory row and widens them to float.
template <typename T, int DL>
struct RowLoad;

template <>
struct RowLoad<F32, 2> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[2]) {
    float2 v = *reinterpret_cast<const float2*>(p);
    o[0] = v.x;
    o[1] = v.y;
  }
};
template <>
struct RowLoad<F32, 4> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
};
template <>
struct RowLoad<BF16, 2> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[2]) {
    uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    o[0] = bf16lo(w);
    o[1] = bf16hi(w);
  }
};
template <>
struct RowLoad<BF16, 4> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    uint2 w = *reinterpret_cast<const uint2*>(p);
    o[0] = bf16lo(w.x);
    o[1] = bf16hi(w.x);
    o[2] = bf16lo(w.y);
    o[3] = bf16hi(w.y);
  }
};
template <>
struct RowLoad<FP8, 2> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[2]) {
    float2 a = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
    o[0] = a.x;
    o[1] = a.y;
  }
};
template <>
struct RowLoad<FP8, 4> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w & 0xffffu));
    float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w >> 16));
    o[0] = a.x;
    o[1] = a.y;
    o[2] = b.x;
    o[3] = b.y;
  }
};

template <>
struct RowLoad<INT8, 2> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[2]) {
    const int8_t* c = reinterpret_cast<const int8_t*>(p);
    o[0] = (float)c[0];
    o[1] = (float)c[1];
  }
};
template <>
struct RowLoad<INT8, 4> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = (float)(int8_t)(w >> (8 * k));
  }
};

__device__ __forceinline__ float load_as_float(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_from_float(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_from_float(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

}  // namespace pkv
