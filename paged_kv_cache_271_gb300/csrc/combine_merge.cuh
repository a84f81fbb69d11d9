// Merge of split-decode partials, shared by the combine kernels of the chunked and the
// balanced decodes. A partial is a running maximum m and sum l (log2 domain) and weighted
// values acc of one (request, query head) over a run of its pages; partials c = lo .. hi - 1
// of one (request, head) sit at ml + 2 c (m, l) and acc + c D (D values). Their merge:
// M = max_c m_c, w_c = 2^(m_c - M), out = sum_c w_c acc_c / sum_c w_c l_c, taken in order c.
#pragma once

#include <math.h>

namespace pkv {

// A warp merges partials lo .. hi - 1 into its running (M, Lw, A), in order: lane L owns dims
// DL L .. DL L + DL - 1 (acc points at the lane's first dim); the (m, l) pairs of up to 32
// partials come in at once (lane c reads partial c's), then the values of CB partials at a
// time; the maximum and the weights go round by shuffles.
template <int D, int CB>
__device__ __forceinline__ void merge_run(const float* ml, const float* acc, int lo, int hi,
                                          int lane, float& M, float& Lw, float (&A)[D / 32]) {
  constexpr int DL = D / 32;
  auto load_batch = [&](int c0, int nc, int cb, float (&v)[CB][DL]) {  // values of CB chunks
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int c = c0 + cb + u;
      if (cb + u < nc) {
        if constexpr (DL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(acc + (size_t)c * D);
          v[u][0] = x.x;
          v[u][1] = x.y;
          v[u][2] = x.z;
          v[u][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(acc + (size_t)c * D);
          v[u][0] = x.x;
          v[u][1] = x.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < DL; ++k) v[u][k] = 0.f;
      }
    }
  };
  for (int c0 = lo; c0 < hi; c0 += 32) {  // 32 chunks per round of (max, sum) pairs
    const int nc = min(32, hi - c0);
    const float2 p = lane < nc ? *reinterpret_cast<const float2*>(ml + 2 * (c0 + lane))
                               : make_float2(-INFINITY, 0.f);
    // the first CB chunks' values do not depend on the pairs: load them together
    float v[CB][DL];
    load_batch(c0, nc, 0, v);
    float mr = p.x;
#pragma unroll
    for (int o = 16; o >= 1; o /= 2) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
    const float Mn = fmaxf(M, mr);
    if (Mn == -INFINITY) continue;
    const float rescale = exp2f(M - Mn);  // 0 on the first round with a finite maximum
    const float w = p.x == -INFINITY ? 0.f : exp2f(p.x - Mn);
    float lw = w * p.y;
#pragma unroll
    for (int o = 16; o >= 1; o /= 2) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    Lw = fmaf(Lw, rescale, lw);
#pragma unroll
    for (int k = 0; k < DL; ++k) A[k] *= rescale;
    M = Mn;
    for (int cb = 0; cb < nc; cb += CB) {
      if (cb > 0) load_batch(c0, nc, cb, v);  // CB chunks' loads in flight together
#pragma unroll
      for (int u = 0; u < CB; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, (cb + u) & 31);
        if (cb + u < nc) {
#pragma unroll
          for (int k = 0; k < DL; ++k) A[k] = fmaf(wu, v[u][k], A[k]);
        }
      }
    }
  }
}

}  // namespace pkv
