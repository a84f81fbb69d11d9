// Write phase (KV append, with optional FP8 quantisation), FP8 scale computation, and the
// split-K combine of decode partials.
//
// kv_append: "KV Cache" glossary, write phase -- the new token's K and V are appended to the
// cache; "KV cache and PagedAttention", section 4 -- they land in a slot of the request's
// page. One thread moves one 16-byte vector of K and the same vector of V; consecutive
// threads cover consecutive dims of one (token, KV head) row, so loads and stores are
// coalesced. FP8: code = cvt.rn.satfinite.e4m3(fp32(x / s)) (section 7, "fp8 KV (E4M3)";
// per-head scale, round-to-nearest-even and saturation are this library's reading).
#include <algorithm>
#include <atomic>
#include <math.h>

#include "combine_merge.cuh"
#include "decode_plan.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

template <typename TIN>
struct Vec16;  // one 16-byte vector of input elements, widened to float
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const void* p, float (&o)[4]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const void* p, float (&o)[8]) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    o[0] = bf16lo(v.x);
    o[1] = bf16hi(v.x);
    o[2] = bf16lo(v.y);
    o[3] = bf16hi(v.y);
    o[4] = bf16lo(v.z);
    o[5] = bf16hi(v.z);
    o[6] = bf16lo(v.w);
    o[7] = bf16hi(v.w);
  }
};

// Same-type append: a straight 16-byte copy per thread.
template <typename T>
__global__ void kv_append_copy_kernel(const AppendArgs a) {
  constexpr int VEC = 16 / sizeof(T);
  const int vpr = a.head_dim / VEC;
  const int64_t total = (int64_t)a.num_tokens * a.h_kv * vpr;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int v = (int)(idx % vpr);
    const int64_t r = idx / vpr;
    const int h = (int)(r % a.h_kv);
    const int64_t i = r / a.h_kv;
    const int64_t slot = a.slots[i];
    if (slot < 0) continue;
    if (slot >= a.num_slots) {
      atomicOr(a.err, PKV_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / kPageSize, row = slot % kPageSize;
    const int64_t src = (i * a.h_kv + h) * a.head_dim + (int64_t)v * VEC;
    const int64_t dst = ((page * a.h_kv + h) * kPageSize + row) * a.head_dim + (int64_t)v * VEC;
    const uint4 kx = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.k_new) + src);
    const uint4 vx = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.v_new) + src);
    *reinterpret_cast<uint4*>(static_cast<T*>(a.k_cache) + dst) = kx;
    *reinterpret_cast<uint4*>(static_cast<T*>(a.v_cache) + dst) = vx;
  }
}

// x / s, correctly rounded to fp32, for a divisor known in advance (the head's scale): with
// r = RN(1/s) computed once, q0 = RN(x r) and one FMA correction q = RN(q0 - r RN(q0 s - x))
// (Markstein's correction step; Brisebarre, Muller and Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance", IEEE Trans. Computers 53(8),
// 2004, study exactly this case). For x with at most 8 significant bits -- every bf16 value --
// and any fp32 s, q equals the IEEE quotient: checked exhaustively over the 2^7 bf16
// significands and the 2^23 fp32 significands of s, which covers every exponent as long as
// no intermediate is subnormal or overflows. That holds for s in [2^-80, 2^80] whenever the
// quotient matters (|q| >= 2^-13; smaller quotients give the code 0 either way). The remainder
// is taken as q0 s - x and subtracted, which equals adding x - q0 s exactly (rounding to
// nearest is symmetric) and keeps the sign of a zero quotient: -0 / s gives -0. Anything else
// -- s outside that range, an infinite or NaN x or an overflow, which all leave a NaN in q --
// takes the IEEE division for the whole vector.
// fp32 inputs (24-bit significands) always take the IEEE division.
struct KnownDivisor {
  float s, r;
  bool fast;
};

__device__ __forceinline__ KnownDivisor known_divisor(float scale) {
  KnownDivisor d;
  d.s = scale;
  d.r = __fdiv_rn(1.f, scale);
  d.fast = scale >= 0x1p-80f && scale <= 0x1p80f;  // (false for NaN)
  return d;
}

// Returns true where the vector took the IEEE division (NaN quotients stay NaN there).
template <typename TIN, int N>
__device__ __forceinline__ bool divide_vec(const float (&x)[N], const KnownDivisor& d,
                                           float (&q)[N]) {
  bool slow = sizeof(TIN) == 4 || !d.fast;
  if (!slow) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const float q0 = __fmul_rn(x[k], d.r);
      q[k] = __fmaf_rn(-__fmaf_rn(q0, d.s, -x[k]), d.r, q0);
      sum = __fadd_rn(sum, q[k]);
    }
    // a NaN quotient makes the sum NaN; so can two infinite ones of opposite signs, which the
    // IEEE division then gives again
    slow = sum != sum;
  }
  if (slow) {
#pragma unroll
    for (int k = 0; k < N; ++k) q[k] = __fdiv_rn(x[k], d.s);
  }
  return slow;
}

template <typename TIN, int N>
__device__ __forceinline__ void quantize_store(const float (&x)[N], const KnownDivisor& d,
                                               uint8_t* dst) {
  float y[N];
  divide_vec<TIN, N>(x, d, y);
  uint16_t codes[N / 2];
#pragma unroll
  for (int k = 0; k < N / 2; ++k)
    codes[k] = static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(y[2 * k], y[2 * k + 1]),
                                                              __NV_SATFINITE, __NV_E4M3));
  if constexpr (N == 8) {
    uint2 w;
    w.x = (uint32_t)codes[0] | ((uint32_t)codes[1] << 16);
    w.y = (uint32_t)codes[2] | ((uint32_t)codes[3] << 16);
    __stcs(reinterpret_cast<uint2*>(dst), w);
  } else {
    __stcs(reinterpret_cast<uint32_t*>(dst), (uint32_t)codes[0] | ((uint32_t)codes[1] << 16));
  }
}

// The INT8 code of y -- y rounded to the nearest integer, ties to even, and clamped to
// [-127, 127] -- in the low byte of the result. Clamping first changes nothing (the bounds are
// integers); adding 1.5 * 2^23 to a value in [-127, 127] gives a sum in [2^23, 2^24), whose
// last significand bit has weight 1, so the addition itself rounds to the nearest integer
// (ties to even: 1.5 * 2^23 is even) and the sum's representation is that of 1.5 * 2^23 plus
// the integer, two's complement in the low bits.
__device__ __forceinline__ uint32_t int8_code_bits(float y) {
  return __float_as_uint(__fadd_rn(fminf(fmaxf(y, -127.f), 127.f), 12582912.f));
}

// INT8 codes of N values: fp32(x / s) rounded to nearest even, clamped to [-127, 127]
// (a NaN quotient gives the code 0).
template <typename TIN, int N>
__device__ __forceinline__ void quantize_store_int8(const float (&x)[N], const KnownDivisor& d,
                                                    uint8_t* dst) {
  float y[N];
  if (divide_vec<TIN, N>(x, d, y)) {
#pragma unroll
    for (int k = 0; k < N; ++k) y[k] = y[k] == y[k] ? y[k] : 0.f;
  }
  uint32_t w[N / 4];
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    // low bytes of four codes into one word: (c0, c1) and (c2, c3), then the two pairs
    const uint32_t c01 = __byte_perm(int8_code_bits(y[4 * k]), int8_code_bits(y[4 * k + 1]),
                                     0x0040);
    const uint32_t c23 = __byte_perm(int8_code_bits(y[4 * k + 2]), int8_code_bits(y[4 * k + 3]),
                                     0x0040);
    w[k] = __byte_perm(c01, c23, 0x5410);
  }
  if constexpr (N == 8) {
    __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
  } else {
    __stcs(reinterpret_cast<uint32_t*>(dst), w[0]);
  }
}

template <typename TIN, bool INT8_CODES>
__device__ __forceinline__ void quantize_vec(const uint4& raw, const KnownDivisor& d,
                                             uint8_t* dst) {
  constexpr int VEC = Vec16<TIN>::N;
  float x[VEC];
  Vec16<TIN>::load(&raw, x);
  if constexpr (INT8_CODES)
    quantize_store_int8<TIN, VEC>(x, d, dst);
  else
    quantize_store<TIN, VEC>(x, d, dst);
}

// Tokens a thread of the quantising append has in flight: their K and V loads are all issued
// before the first store (measured on a 25,032-token prompt batch: 1 and 2 tokens about the
// same, 4 and 8 slower). Rows are read and codes written with evict-first hints: each byte is
// touched once here.
constexpr int kAppendTokens = 2;

// FP8 / INT8 append: each 16-byte vector of fp32/bf16 input is quantised with its head's scale
// and its codes stored at the token's slot. A thread owns fixed (head, vector) columns of the
// token rows -- their index arithmetic and scales are set once -- and walks the tokens
// blockIdx.x, blockIdx.x + gridDim.x, ..., kAppendTokens at a time.
template <typename TIN, bool INT8_CODES>
__global__ void kv_append_fp8_kernel(const AppendArgs a) {
  constexpr int VEC = Vec16<TIN>::N;
  constexpr int U = kAppendTokens;
  const int vpr = a.head_dim / VEC;
  const int per_tok = a.h_kv * vpr;
  const int64_t row_elems = (int64_t)a.h_kv * a.head_dim;  // one token's input row
  const int64_t page_elems = row_elems * kPageSize;        // one pool page (every head)
  const TIN* kin = static_cast<const TIN*>(a.k_new);
  const TIN* vin = static_cast<const TIN*>(a.v_new);
  uint8_t* kc = static_cast<uint8_t*>(a.k_cache);
  uint8_t* vc = static_cast<uint8_t*>(a.v_cache);
  const int n = a.num_tokens, step = gridDim.x;
  for (int t = threadIdx.x; t < per_tok; t += blockDim.x) {
    const int h = t / vpr, v = t - h * vpr;
    const KnownDivisor ks = known_divisor(a.k_scales[h]), vs = known_divisor(a.v_scales[h]);
    const int64_t src0 = (int64_t)h * a.head_dim + v * VEC;
    const int64_t dst0 = (int64_t)h * kPageSize * a.head_dim + v * VEC;
    for (int i = blockIdx.x; i < n; i += U * step) {
      int64_t slot[U];
      uint4 kx[U], vx[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int iu = i + u * step;
        slot[u] = -1;
        kx[u] = vx[u] = make_uint4(0, 0, 0, 0);
        if (iu < n) {
          slot[u] = a.slots[iu];
          kx[u] = __ldcs(reinterpret_cast<const uint4*>(kin + iu * row_elems + src0));
          vx[u] = __ldcs(reinterpret_cast<const uint4*>(vin + iu * row_elems + src0));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t sl = slot[u];
        if (sl >= a.num_slots) atomicOr(a.err, PKV_DEVERR_BAD_SLOT);
        if (sl >= 0 && sl < a.num_slots) {
          const int64_t d = (sl / kPageSize) * page_elems + (sl % kPageSize) * a.head_dim + dst0;
          quantize_vec<TIN, INT8_CODES>(kx[u], ks, kc + d);
          quantize_vec<TIN, INT8_CODES>(vx[u], vs, vc + d);
        }
      }
    }
  }
}

// max |x| per KV head: grid.y = head; bits of the non-negative float maximum are combined with
// an integer atomicMax (order-preserving for non-negative floats).
template <typename TIN>
__global__ void kv_absmax_kernel(const TIN* x, int64_t n_tokens, int h_kv, int head_dim,
                                 unsigned int* bits) {
  constexpr int VEC = Vec16<TIN>::N;
  const int h = blockIdx.y;
  const int vpr = head_dim / VEC;
  const int64_t total = n_tokens * vpr;
  float m = 0.f;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / vpr;
    const int v = (int)(e % vpr);
    float xs[VEC];
    Vec16<TIN>::load(x + (t * h_kv + h) * head_dim + (int64_t)v * VEC, xs);
#pragma unroll
    for (int k = 0; k < VEC; ++k) m = fmaxf(m, fabsf(xs[k]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float bm = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) bm = fmaxf(bm, wmax[w]);
    atomicMax(bits + h, __float_as_uint(bm));
  }
}

__global__ void kv_scale_finalize_kernel(float* scales, int h_kv, float code_max) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= h_kv) return;
  const float amax = __uint_as_float(reinterpret_cast<unsigned int*>(scales)[h]);
  scales[h] = (amax == 0.f) ? 1.f : __fdiv_rn(amax, code_max);
}

// Merge of the chunk partials of one (b, h) in chunk order (merge_run). Launched as a
// programmatic dependent of the decode kernel, whose CTAs allow
// it to be scheduled as they start: its CTAs are placed while the decode's last CTAs run and
// wait for the decode's results before reading them.
//  * few chunks (SPLIT false): one warp per (h, b), four per CTA, no block barrier;
//  * many chunks (SPLIT true, a long context cut into up to hundreds of chunks): one CTA per
//    (h, b) whose four warps each merge a quarter of the chunks (a run of consecutive chunks),
//    then warp 0 merges the four results in warp order, so fewer loads wait on one another.
template <typename TQ, int D, bool SPLIT>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a) {
  constexpr int DL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = SPLIT ? blockIdx.x : blockIdx.x * 4 + warp, b = blockIdx.y;
  if (h >= a.h_q) return;
  // the chunk count depends on inputs only: known before the decode's results are
  const int ctx = min(max(0, a.context_lens[b]), a.max_pages * kPageSize);
  const int n_chunks = seq_plan(a, b, ctx).n_total;  // partials of the request
  if (n_chunks <= 1) return;  // (uniform over the CTA when SPLIT)
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid is done, its writes seen
  const size_t bh = (size_t)b * a.h_q + h;
  const float* ml = a.ws_ml + bh * a.n_chunk_slots * 2;
  const float* acc = a.ws_acc + bh * a.n_chunk_slots * D + lane * DL;

  float M = -INFINITY, Lw = 0.f, A[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) A[k] = 0.f;
  if constexpr (!SPLIT) {
    merge_run<D, 8>(ml, acc, 0, n_chunks, lane, M, Lw, A);
  } else {
    const int q = (n_chunks + 3) / 4;
    merge_run<D, 16>(ml, acc, min(n_chunks, warp * q), min(n_chunks, (warp + 1) * q), lane, M,
                     Lw, A);
    __shared__ float red_a[4][D];
    __shared__ float red_ml[4][2];
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
  }
#pragma unroll
  for (int k = 0; k < DL; ++k)
    store_from_float(static_cast<TQ*>(a.out), bh * D + lane * DL + k, Lw > 0.f ? A[k] / Lw : 0.f);
}

// Chunk slots above which one CTA (four warps) merges each (request, head)
constexpr int kCombineSplitSlots = 16;

template <typename TQ, int D>
cudaError_t launch_combine_t(const DecodeArgs& a, cudaStream_t s) {
  const bool split = a.n_chunk_slots > kCombineSplitSlots;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split ? a.h_q : (a.h_q + 3) / 4, a.batch);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return split ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<TQ, D, true>, a)
               : cudaLaunchKernelEx(&cfg, decode_combine_kernel<TQ, D, false>, a);
}

// Copy whole pages (every KV head's tile) of both pools: pool[dst[p]] = pool[src[p]]. One
// thread moves 16 bytes of K and the same 16 bytes of V. Out-of-range ids are skipped and
// flagged as bad pages.
__global__ void copy_pages_kernel(uint8_t* k, uint8_t* v, const int32_t* src, const int32_t* dst,
                                  int n, int64_t page_bytes, int num_pages, int* err) {
  const int64_t vecs = page_bytes / 16;
  const int64_t total = (int64_t)n * vecs;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx / vecs);
    const int64_t off = (idx % vecs) * 16;
    const int s = src[p], d = dst[p];
    if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
      atomicOr(err, PKV_DEVERR_BAD_PAGE);
      continue;
    }
    *reinterpret_cast<uint4*>(k + d * page_bytes + off) =
        *reinterpret_cast<const uint4*>(k + s * page_bytes + off);
    *reinterpret_cast<uint4*>(v + d * page_bytes + off) =
        *reinterpret_cast<const uint4*>(v + s * page_bytes + off);
  }
}

inline int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, int in_dtype, int cache_dtype, cudaStream_t s) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  if (cache_dtype == PKV_FP8_E4M3 || cache_dtype == PKV_INT8) {
    const bool i8 = cache_dtype == PKV_INT8;
    // one wave of blocks, each taking kAppendTokens tokens at a time; threads cover a token
    // row's (head, vector) columns
    const int per_tok = a.h_kv * (a.head_dim / (in_dtype == PKV_BF16 ? 8 : 4));
    const int qt = per_tok <= 128 ? 128 : 256;
    const int64_t groups = ((int64_t)a.num_tokens + kAppendTokens - 1) / kAppendTokens;
    auto go = [&](auto kern, int slot) {
      static std::atomic<int> wave[2];  // resident blocks on the device, per block size
      if (!wave[slot].load()) {
        int per_sm = 0, dev = 0, sms = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, qt, 0);
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        wave[slot].store(std::max(1, per_sm) * std::max(1, sms));
      }
      const int blocks = (int)std::min<int64_t>(groups, wave[slot].load());
      kern<<<blocks, qt, 0, s>>>(a);
    };
    const int slot = qt == 128 ? 0 : 1;
    if (in_dtype == PKV_BF16) {
      if (i8)
        go(kv_append_fp8_kernel<__nv_bfloat16, true>, slot);
      else
        go(kv_append_fp8_kernel<__nv_bfloat16, false>, slot);
    } else {
      if (i8)
        go(kv_append_fp8_kernel<float, true>, slot);
      else
        go(kv_append_fp8_kernel<float, false>, slot);
    }
  } else if (cache_dtype == PKV_BF16) {
    const int64_t work = (int64_t)a.num_tokens * a.h_kv * (a.head_dim / 8);
    kv_append_copy_kernel<__nv_bfloat16><<<grid_for(work, threads), threads, 0, s>>>(a);
  } else {
    const int64_t work = (int64_t)a.num_tokens * a.h_kv * (a.head_dim / 4);
    kv_append_copy_kernel<float><<<grid_for(work, threads), threads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_absmax(const void* x, int dtype, int64_t n_tokens, int h_kv, int head_dim,
                             float code_max, float* scales_out, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(scales_out, 0, sizeof(float) * h_kv, s);
  if (e != cudaSuccess) return e;
  if (n_tokens > 0) {
    const int threads = 256;
    const int vec = dtype == PKV_BF16 ? 8 : 4;
    const int64_t work = n_tokens * (head_dim / vec);
    int bx = grid_for(work, threads);
    const int cap = (152 * 8 + h_kv - 1) / h_kv;
    if (bx > cap) bx = cap < 1 ? 1 : cap;
    dim3 grid(bx, h_kv);
    unsigned int* bits = reinterpret_cast<unsigned int*>(scales_out);
    if (dtype == PKV_BF16)
      kv_absmax_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
          static_cast<const __nv_bfloat16*>(x), n_tokens, h_kv, head_dim, bits);
    else
      kv_absmax_kernel<float><<<grid, threads, 0, s>>>(static_cast<const float*>(x), n_tokens,
                                                       h_kv, head_dim, bits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  kv_scale_finalize_kernel<<<(h_kv + 127) / 128, 128, 0, s>>>(scales_out, h_kv, code_max);
  return cudaGetLastError();
}

cudaError_t launch_copy_pages(void* k, void* v, const int32_t* src, const int32_t* dst, int n,
                              int64_t page_bytes, int num_pages, int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  copy_pages_kernel<<<grid_for((int64_t)n * (page_bytes / 16), threads), threads, 0, s>>>(
      static_cast<uint8_t*>(k), static_cast<uint8_t*>(v), src, dst, n, page_bytes, num_pages,
      err);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeArgs& a, int q_dtype, int head_dim, cudaStream_t s) {
  if (q_dtype == PKV_BF16)
    return head_dim == 64 ? launch_combine_t<__nv_bfloat16, 64>(a, s)
                          : launch_combine_t<__nv_bfloat16, 128>(a, s);
  return head_dim == 64 ? launch_combine_t<float, 64>(a, s) : launch_combine_t<float, 128>(a, s);
}

}  // namespace pkv
