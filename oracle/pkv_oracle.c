/*
 * CPU oracle for single-token decode attention over a paged KV cache -- TEST INFRASTRUCTURE.
 *
 * This file is the slow, plain, fp64 statement of what the CUDA library computes. It is used
 * only by the tests, by the smoke check and by the benchmark's CPU-baseline leg; nothing on
 * the product path may link or call it. It shares no code, header or table with the CUDA
 * library.
 *
 * What it follows (the KV-cache pages):
 *  - "KV cache and PagedAttention", section 1 (The setup): at each decode step only the new
 *    token's query is used; attention reads the whole cached K and V (cached + new).
 *  - "Memoizing Context via KV Caching": the query is compared with every cached key to form
 *    attention weights, which then weight a sum of the value vectors (softmax attention).
 *  - "KV cache and PagedAttention", section 4: the cache is a pool of fixed-size pages; a
 *    per-request page table lists page indices; attention gathers K/V through that table.
 *  - "KV Cache" glossary, GQA / MQA paragraphs: several query heads share one KV head.
 *    Reading taken (the pages give no order): query head h uses KV head h / (h_q / h_kv).
 *  - "KV cache and PagedAttention", section 7: an FP8 E4M3 cache. The code values follow the
 *    OCP 8-bit floating point specification (E4M3: bias 7, no infinities, S.1111.111 is NaN,
 *    largest finite 448). Readings taken: one fp32 scale per (layer, kv head), value = code
 *    value * scale; quantisation = fp32 division by the scale, then round to nearest even
 *    with saturation to +-448.
 *
 * Pool layout read here: [num_pages][h_kv][page_size][d] (one contiguous tile per page and
 * KV head); token t of a request lives in page block_table[t / page_size] at row
 * t % page_size. Every stored value is converted to double exactly before use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_INT8 = 3 };

/* ---- OCP FP8 E4M3 ------------------------------------------------------------------- */

/* Value of one E4M3 code: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 encodes subnormals 0.m * 2^-6; field 15 with mantissa 7 is NaN. */
double oracle_e4m3_value(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest E4M3 code to y: round to nearest, ties to the even code (the code's lowest bit is
 * the mantissa's lowest bit), saturating to the largest finite magnitude 448 for anything
 * at or beyond it. The non-negative finite codes 0x00..0x7E are ordered by value, so the
 * neighbours of |y| are found by bisection over that table. NaN stays NaN; the sign of y
 * (also of a zero result) is kept. */
uint8_t oracle_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_value((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double dlo = a - oracle_e4m3_value((uint8_t)lo);
  double dhi = oracle_e4m3_value((uint8_t)hi) - a;
  int pick;
  if (dlo < dhi)
    pick = lo;
  else if (dhi < dlo)
    pick = hi;
  else
    pick = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | pick);
}

/* out[i] = encode(fp32(x[i] / s)): the division is IEEE binary32, rounded to nearest. */
void oracle_quantize_e4m3(const float* x, int64_t n, float s, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    float y = x[i] / s;
    out[i] = oracle_e4m3_encode(y);
  }
}

/* ---- INT8 ------------------------------------------------------------------------------- */

/* "INT8 KV" ("KV cache and PagedAttention", section 7) with the reading taken here: a
 * symmetric code c in [-127, 127], value = c * scale, code = fp32(x / scale) rounded to the
 * nearest integer (ties to even) and clamped to [-127, 127]. Inputs are finite. */
void oracle_quantize_int8(const float* x, int64_t n, float s, int8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    float y = x[i] / s;
    double r = nearbyint((double)y); /* default rounding mode: to nearest, ties to even */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    out[i] = (int8_t)r;
  }
}

/* ---- exact element reads --------------------------------------------------------------- */

static double bf16_value(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double read_elem(const void* base, int dtype, int64_t idx, double code_scale) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[idx];
    case ORC_BF16: return bf16_value(((const uint16_t*)base)[idx]);
    case ORC_INT8: return (double)((const int8_t*)base)[idx] * code_scale;
    default: return oracle_e4m3_value(((const uint8_t*)base)[idx]) * code_scale;
  }
}

/* ---- attention -------------------------------------------------------------------------- */

/* Tokens attended by a request of T tokens ("KV cache and PagedAttention", section 8): with a
 * sliding window of W tokens only the last W are kept; with S attention sinks the first S are
 * kept as well. W == 0 means no window (every token). */
static int attended(int64_t t, int64_t T, int sink, int window) {
  if (window <= 0) return 1;
  return t >= T - window || t < sink;
}

/* Textbook softmax attention of one query over T keys/values, all in double:
 *   x_t = scale * <q, K_t>,  p_t = exp(x_t - max x) / sum_u exp(x_u - max x),
 *   out = sum_t p_t V_t.
 * K and V are supplied as gathered double rows [T][d]. T == 0 gives out = 0. */
void oracle_attend(const double* q, const double* K, const double* V, int64_t T, int d,
                   double scale, double* out) {
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  if (T <= 0) return;
  double* x = (double*)malloc((size_t)T * sizeof(double));
  double mx = -INFINITY;
  for (int64_t t = 0; t < T; ++t) {
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += q[i] * K[t * d + i];
    x[t] = scale * dot;
    if (x[t] > mx) mx = x[t];
  }
  double den = 0.0;
  for (int64_t t = 0; t < T; ++t) {
    x[t] = exp(x[t] - mx);
    den += x[t];
  }
  for (int64_t t = 0; t < T; ++t)
    for (int i = 0; i < d; ++i) out[i] += (x[t] / den) * V[t * d + i];
  free(x);
}

/* Gather the keys and values of request b, KV head j, through its page table:
 * token t is row t % P of page block_tables[b][t / P]. Returns -1 on an out-of-range page. */
static int gather_paged(const void* k_pool, const void* v_pool, int kv_dtype, int num_pages,
                        int h_kv, int P, int d, const int32_t* bt_row, int64_t T, int j,
                        double ks, double vs, double* K, double* V, int sink, int window) {
  int64_t n = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (!attended(t, T, sink, window)) continue; /* its page need not exist any more */
    int32_t page = bt_row[t / P];
    if (page < 0 || page >= num_pages) return -1;
    int64_t row = ((int64_t)page * h_kv + j) * P + (t % P);
    for (int i = 0; i < d; ++i) {
      K[n * d + i] = read_elem(k_pool, kv_dtype, row * d + i, ks);
      V[n * d + i] = read_elem(v_pool, kv_dtype, row * d + i, vs);
    }
    ++n;
  }
  return 0;
}

/* Decode attention over a paged pool for the listed (b, h) pairs (all pairs when pairs is
 * NULL). out rows follow the pair order: out[k][d] for pair k, or out[b][h][d] for all.
 * sink/window select the attended tokens as in attended() (window 0: all); pages holding no
 * attended token are not read. Returns 0, or -1 if a page id it reads is out of range (that
 * pair's output is left at 0). */
int oracle_paged_decode(const void* q, int q_dtype, int B, int h_q, int d, const void* k_pool,
                        const void* v_pool, int kv_dtype, int num_pages, int h_kv, int P,
                        const int32_t* block_tables, int max_pages, const int32_t* context_lens,
                        double scale, const float* k_scales, const float* v_scales,
                        const int32_t* pairs, int n_pairs, double* out, int n_threads,
                        int sink, int window) {
  int G = h_q / h_kv;
  int total = pairs ? n_pairs : B * h_q;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
#endif
  for (int k = 0; k < total; ++k) {
    int b = pairs ? pairs[2 * k] : k / h_q;
    int h = pairs ? pairs[2 * k + 1] : k % h_q;
    int j = h / G;
    int64_t T = context_lens[b];
    double ks = (kv_dtype >= ORC_E4M3) ? (double)k_scales[j] : 1.0;
    double vs = (kv_dtype >= ORC_E4M3) ? (double)v_scales[j] : 1.0;
    double* qd = (double*)malloc((size_t)d * sizeof(double));
    double* K = (double*)malloc((size_t)(T > 0 ? T : 1) * d * sizeof(double));
    double* V = (double*)malloc((size_t)(T > 0 ? T : 1) * d * sizeof(double));
    for (int i = 0; i < d; ++i)
      qd[i] = read_elem(q, q_dtype, ((int64_t)b * h_q + h) * d + i, 1.0);
    if (gather_paged(k_pool, v_pool, kv_dtype, num_pages, h_kv, P, d,
                     block_tables + (int64_t)b * max_pages, T, j, ks, vs, K, V, sink,
                     window) != 0) {
      for (int i = 0; i < d; ++i) out[(int64_t)k * d + i] = 0.0;
      status = -1;
    } else {
      int64_t n = 0; /* attended tokens, packed to the front by the gather */
      for (int64_t t = 0; t < T; ++t) n += attended(t, T, sink, window);
      oracle_attend(qd, K, V, n, d, scale, out + (int64_t)k * d);
    }
    free(qd);
    free(K);
    free(V);
  }
  return status;
}

/* Decode attention over contiguous (un-paged) per-request keys and values: request b's token
 * t, KV head j, is row (offsets[b] + t) of kv[rows][h_kv][d]. When prefix_len > 0, tokens
 * t < prefix_len come from prefix_k/prefix_v[prefix_len][h_kv][d] instead and the request's
 * own rows start at offsets[b] for t = prefix_len. This is the naive cache ("KV cache and
 * PagedAttention", section 3) that the paged layout must reproduce. sink/window select the
 * attended tokens as in attended() (window 0: all). */
int oracle_contiguous_decode(const void* q, int q_dtype, int B, int h_q, int d, const void* k_rows,
                             const void* v_rows, const void* prefix_k, const void* prefix_v,
                             int prefix_len, int kv_dtype, int h_kv, const int64_t* offsets,
                             const int32_t* context_lens, double scale, const float* k_scales,
                             const float* v_scales, const int32_t* pairs, int n_pairs,
                             double* out, int n_threads, int sink, int window) {
  int G = h_q / h_kv;
  int total = pairs ? n_pairs : B * h_q;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int k = 0; k < total; ++k) {
    int b = pairs ? pairs[2 * k] : k / h_q;
    int h = pairs ? pairs[2 * k + 1] : k % h_q;
    int j = h / G;
    int64_t T = context_lens[b];
    double ks = (kv_dtype >= ORC_E4M3) ? (double)k_scales[j] : 1.0;
    double vs = (kv_dtype >= ORC_E4M3) ? (double)v_scales[j] : 1.0;
    double* qd = (double*)malloc((size_t)d * sizeof(double));
    double* K = (double*)malloc((size_t)(T > 0 ? T : 1) * d * sizeof(double));
    double* V = (double*)malloc((size_t)(T > 0 ? T : 1) * d * sizeof(double));
    for (int i = 0; i < d; ++i)
      qd[i] = read_elem(q, q_dtype, ((int64_t)b * h_q + h) * d + i, 1.0);
    int64_t n = 0; /* attended tokens, in order */
    for (int64_t t = 0; t < T; ++t) {
      if (!attended(t, T, sink, window)) continue;
      for (int i = 0; i < d; ++i) {
        if (t < prefix_len) {
          int64_t idx = (t * h_kv + j) * d + i;
          K[n * d + i] = read_elem(prefix_k, kv_dtype, idx, ks);
          V[n * d + i] = read_elem(prefix_v, kv_dtype, idx, vs);
        } else {
          int64_t idx = ((offsets[b] + t - prefix_len) * h_kv + j) * d + i;
          K[n * d + i] = read_elem(k_rows, kv_dtype, idx, ks);
          V[n * d + i] = read_elem(v_rows, kv_dtype, idx, vs);
        }
      }
      ++n;
    }
    oracle_attend(qd, K, V, n, d, scale, out + (int64_t)k * d);
    free(qd);
    free(K);
    free(V);
  }
  return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
