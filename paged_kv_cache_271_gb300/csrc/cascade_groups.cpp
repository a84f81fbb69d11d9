// Host side of the cascade decode: finds the requests of a batch whose page tables start with
// the same physical pages -- the pages of a shared prompt prefix ("KV cache and
// PagedAttention", section 6) -- and describes them as groups for the prefix kernel.
//
// Requests are bucketed by their first page id in batch order; a bucket of at least
// min_members requests becomes a group sharing the longest run of leading page ids common to
// all its members, cut so that every member's context reaches past it (the page holding
// position ctx - 1, which a decode step writes, is never shared). A group sharing fewer than
// min_prefix_pages pages is dropped. Members keep batch order inside their group.
#include <algorithm>
#include <cstring>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"

namespace {

// Per-thread scratch of the grouping, kept across calls so that a call allocates nothing once
// the batch size has been seen: an open-addressing table from first page id to bucket (a slot
// is live when its stamp equals the call's epoch, so the table is never cleared), and the
// bucket arrays.
struct GroupScratch {
  std::vector<int32_t> key, val;
  std::vector<uint32_t> stamp;
  uint32_t epoch = 0;
  std::vector<int32_t> bucket, count, start, flat, fill;
};
thread_local GroupScratch t_scratch;

}  // namespace

extern "C" int pkv_cascade_groups(const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t batch, int32_t max_pages_per_seq, int32_t min_members,
                                  int32_t min_prefix_pages, int32_t* group_of,
                                  int32_t* prefix_pages, int32_t* group_offsets,
                                  int32_t* group_members, int32_t* n_groups,
                                  int32_t* max_members, int32_t* max_prefix_pages,
                                  int32_t* max_own_pages, int32_t* own_start) {
  if (batch < 0 || max_pages_per_seq <= 0 || (batch > 0 && (!block_tables || !context_lens ||
      !group_of || !prefix_pages || !group_members)) || !group_offsets || !n_groups ||
      !max_members || !max_prefix_pages || !max_own_pages)
    return pkv::set_error(PKV_EINVAL, "pkv_cascade_groups: bad argument");
  if (min_members < 2) min_members = 2;
  if (min_prefix_pages < 1) min_prefix_pages = 1;
  const int32_t P = 16;
  // pages every member may share: the full pages before the one holding position ctx - 1
  auto cap = [&](int b) {
    const int64_t ctx = context_lens[b];
    const int64_t c = ctx >= 1 ? (ctx - 1) / P : 0;
    return (int32_t)std::min<int64_t>(c, max_pages_per_seq);
  };
  // bucket of each request (by first page id, buckets numbered in order of first appearance),
  // then the members of every bucket in batch order, in one flat array (a counting pass)
  GroupScratch& w = t_scratch;
  size_t slots = 16;
  while (slots < (size_t)batch * 2) slots *= 2;
  if (w.key.size() < slots) {
    w.key.assign(slots, 0);
    w.val.assign(slots, 0);
    w.stamp.assign(slots, 0);
    w.epoch = 0;
  }
  if (++w.epoch == 0) {  // the stamps wrapped: forget them all once
    std::fill(w.stamp.begin(), w.stamp.end(), 0u);
    w.epoch = 1;
  }
  const size_t mask = slots - 1;
  w.bucket.assign(batch, -1);
  w.count.clear();
  for (int32_t b = 0; b < batch; ++b) {
    group_of[b] = -1;
    if (cap(b) < min_prefix_pages) continue;
    const int32_t first = block_tables[(size_t)b * max_pages_per_seq];
    size_t i = ((uint32_t)first * 2654435761u) & mask;  // multiplicative hash, linear probing
    while (w.stamp[i] == w.epoch && w.key[i] != first) i = (i + 1) & mask;
    if (w.stamp[i] != w.epoch) {  // a new first page: the next bucket
      w.stamp[i] = w.epoch;
      w.key[i] = first;
      w.val[i] = (int32_t)w.count.size();
      w.count.push_back(0);
    }
    w.bucket[b] = w.val[i];
    ++w.count[w.bucket[b]];
  }
  const std::vector<int32_t>& bucket = w.bucket;
  const std::vector<int32_t>& count = w.count;
  const int32_t nb = (int32_t)count.size();
  std::vector<int32_t>& start = w.start;
  start.assign(nb + 1, 0);
  for (int32_t k = 0; k < nb; ++k) start[k + 1] = start[k] + count[k];
  std::vector<int32_t>& flat = w.flat;
  flat.resize(start[nb]);
  w.fill.assign(start.begin(), start.end() - 1);
  for (int32_t b = 0; b < batch; ++b)
    if (bucket[b] >= 0) flat[w.fill[bucket[b]]++] = b;
  int32_t ng = 0, nm = 0, mm = 0, mp = 0;
  group_offsets[0] = 0;
  for (int32_t k = 0; k < nb; ++k) {
    const int32_t* mem = flat.data() + start[k];
    const int32_t size = count[k];
    if (size < min_members) continue;
    const int32_t* r0 = block_tables + (size_t)mem[0] * max_pages_per_seq;
    int32_t shared = cap(mem[0]);
    for (int32_t m = 1; m < size && shared > 0; ++m) {
      const int32_t* r = block_tables + (size_t)mem[m] * max_pages_per_seq;
      const int32_t lim = std::min(shared, cap(mem[m]));
      int32_t n = lim;
      if (std::memcmp(r, r0, (size_t)lim * sizeof(int32_t)) != 0) {  // find where they part
        n = 0;
        while (r[n] == r0[n]) ++n;
      }
      shared = n;
    }
    if (shared < min_prefix_pages) continue;
    for (int32_t m = 0; m < size; ++m) {
      group_of[mem[m]] = ng;
      group_members[nm++] = mem[m];
    }
    prefix_pages[ng] = shared;
    group_offsets[ng + 1] = nm;
    mm = std::max(mm, size);
    mp = std::max(mp, shared);
    ++ng;
  }
  int32_t mo = 0;  // pages each request reads itself
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t ctx = std::min<int64_t>(std::max(context_lens[b], 0), (int64_t)P * max_pages_per_seq);
    const int32_t pages = (int32_t)((ctx + P - 1) / P);
    const int32_t start = group_of[b] >= 0 ? prefix_pages[group_of[b]] : 0;
    mo = std::max(mo, pages - start);
    if (own_start) own_start[b] = start;
  }
  *n_groups = ng;
  *max_members = mm;
  *max_prefix_pages = mp;
  *max_own_pages = mo;
  return PKV_OK;
}

extern "C" int pkv_cascade_prefix_page_ids(const int32_t* block_tables, int32_t batch,
                                           int32_t max_pages_per_seq,
                                           const int32_t* prefix_pages,
                                           const int32_t* group_offsets,
                                           const int32_t* group_members, int32_t n_groups,
                                           int32_t max_prefix_pages, int32_t* ids_out) {
  if (n_groups < 0 || batch < 0 || max_prefix_pages < 0 ||
      max_prefix_pages > max_pages_per_seq ||
      (n_groups > 0 && (!block_tables || !prefix_pages || !group_offsets || !group_members ||
                        !ids_out)))
    return pkv::set_error(PKV_EINVAL, "pkv_cascade_prefix_page_ids: bad argument");
  for (int32_t g = 0; g < n_groups; ++g) {
    const int32_t pp = prefix_pages[g];
    const int32_t first = group_offsets[g] < group_offsets[g + 1] && group_offsets[g] >= 0
                              ? group_members[group_offsets[g]]
                              : -1;
    if (pp < 0 || pp > max_prefix_pages || first < 0 || first >= batch)
      return pkv::set_error(PKV_EINVAL, "pkv_cascade_prefix_page_ids: group %d is malformed", g);
    const int32_t* row = block_tables + (size_t)first * max_pages_per_seq;
    int32_t* out = ids_out + (size_t)g * max_prefix_pages;
    std::memcpy(out, row, (size_t)pp * sizeof(int32_t));
    for (int32_t i = pp; i < max_prefix_pages; ++i) out[i] = -1;
  }
  return PKV_OK;
}
