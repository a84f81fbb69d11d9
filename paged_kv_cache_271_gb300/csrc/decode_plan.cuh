// Which logical pages of request b one decode launch reads, and where their partial results
// go; shared by both decode kernels and the combine kernel so that all three agree.
//
// Plain decode: the attended pages (all of them, or the sink and window pages), split into
// the fewest near-equal chunks of at most chunk_pages pages, one CTA each; one chunk writes
// the output directly, several write partials to chunk slots 0, 1, ... for the combine.
//
// Cascade decode (a request in a group that shares its first P logical pages with the other
// members, "KV cache and PagedAttention" section 6): the prefix kernel covers those P pages
// once for the whole group and writes its partials to slots 0 .. ceil(P / prefix_chunk_pages)
// - 1 of every member; the decode kernel then reads pages P .. of the request only and its
// chunks write their partials after the prefix's (slots slot0 ..). Who merges: by default the
// combine kernel, which merges all of a request's slots; or (overlap modes 0 and 1) the decode
// kernel itself -- a single own chunk (possibly empty) folds the prefix partials in and writes
// the output, and with several the last chunk to finish merges them all.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct SeqPlan {
  SeqPages sp;   // the pages this decode reads, in logical order
  int slot0;     // chunk slot of the first of its partials
  int n_chunks;  // chunks (CTAs) over sp
  int n_total;   // partials merged for the request; <= 1: the decode writes the output
  int prefix;    // shared prefix pages handled by the prefix kernel (0: none)
};

__device__ __forceinline__ int cascade_prefix_chunks(const DecodeArgs& a, int prefix_pages) {
  return prefix_pages > 0 ? (prefix_pages + a.prefix_chunk_pages - 1) / a.prefix_chunk_pages : 0;
}

// Shared prefix pages of group g as the kernels use them (clamped to what the launch declared).
__device__ __forceinline__ int cascade_group_pages(const DecodeArgs& a, int g) {
  return min(max(0, a.prefix_pages[g]), a.max_prefix_pages);
}

__device__ __forceinline__ SeqPlan seq_plan(const DecodeArgs& a, int b, int ctx) {
  SeqPlan p;
  p.sp = seq_pages(ctx, a.sink, a.window);
  p.slot0 = 0;
  p.prefix = 0;
  if (a.group_of != nullptr) {
    int pp = 0;
    if (a.own_start != nullptr) {  // the member's shared pages, without the group lookup
      pp = min(max(0, a.own_start[b]), a.max_prefix_pages);
    } else {
      const int g = a.group_of[b];
      if (g >= 0 && g < a.n_groups) pp = cascade_group_pages(a, g);
    }
    if (pp > 0) {  // no window in a cascade decode: sp covers pages 0 .. n-1
      p.prefix = pp;
      p.sp = SeqPages{max(0, p.sp.n - pp), 0, pp};
      p.slot0 = cascade_prefix_chunks(a, pp);
    }
  }
  // the grid has chunk_grid chunk columns: a longer run of pages takes larger chunks
  p.n_chunks = min((p.sp.n + a.chunk_pages - 1) / a.chunk_pages, a.chunk_grid);
  p.n_total = p.slot0 > 0 ? p.slot0 + max(p.n_chunks, 1) : p.n_chunks;
  return p;
}

}  // namespace pkv
