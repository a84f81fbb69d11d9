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
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"

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
  std::unordered_map<int32_t, int32_t> bucket_of;  // first page id -> bucket
  std::vector<std::vector<int32_t>> buckets;
  for (int32_t b = 0; b < batch; ++b) {
    group_of[b] = -1;
    if (cap(b) < min_prefix_pages) continue;
    const int32_t first = block_tables[(size_t)b * max_pages_per_seq];
    auto it = bucket_of.find(first);
    if (it == bucket_of.end()) {
      bucket_of.emplace(first, (int32_t)buckets.size());
      buckets.push_back({b});
    } else {
      buckets[it->second].push_back(b);
    }
  }
  int32_t ng = 0, nm = 0, mm = 0, mp = 0;
  group_offsets[0] = 0;
  for (const auto& mem : buckets) {
    if ((int32_t)mem.size() < min_members) continue;
    const int32_t* r0 = block_tables + (size_t)mem[0] * max_pages_per_seq;
    int32_t shared = cap(mem[0]);
    for (size_t k = 1; k < mem.size() && shared > 0; ++k) {
      const int32_t* r = block_tables + (size_t)mem[k] * max_pages_per_seq;
      int32_t n = 0;
      const int32_t lim = std::min(shared, cap(mem[k]));
      while (n < lim && r[n] == r0[n]) ++n;
      shared = n;
    }
    if (shared < min_prefix_pages) continue;
    for (int32_t b : mem) {
      group_of[b] = ng;
      group_members[nm++] = b;
    }
    prefix_pages[ng] = shared;
    group_offsets[ng + 1] = nm;
    mm = std::max(mm, (int32_t)mem.size());
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
