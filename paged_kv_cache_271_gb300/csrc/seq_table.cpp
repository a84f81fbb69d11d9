// Per-request page tables over the page allocator ("KV cache and PagedAttention", section 4:
// each request keeps a list of the pages holding its tokens; section 5: requests join and
// leave every step; section 6 and the "KV Cache" glossary: prompt prefixes, parallel samples
// and beams share pages, a shared page being copied before its first divergent write; section
// 8: pages wholly outside a sliding window go back to the pool).
//
// A request is a row of page ids (-1 where a page was released) and a token count. Every page
// in a row holds one reference of the allocator, so sharing is counting: a fork takes one more
// reference on each of the parent's pages, freeing a request drops its references. Reserving
// n more tokens for a request first copies-on-write the page its next token lands in when that
// page is shared and partly filled (the pair to copy is returned, the device copy is the
// caller's), then allocates the pages the new length needs, and returns each new token's slot
// page * P + offset. A reserve checks, before it changes anything, that the free pages cover
// every copy and page it will take (replaying the reference counts in batch order), so it
// either completes or changes nothing.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"

namespace {

struct Seq {
  std::vector<int32_t> pages;  // -1: released (outside a window)
  int64_t len = 0;
  uint64_t mark = 0;  // the table's epoch of the last batch call that listed it
};

int64_t pages_for(int64_t tokens, int32_t P) { return (tokens + P - 1) / P; }

}  // namespace

struct pkv_seq_table {
  pkv_allocator* alloc;
  int32_t page_size;
  std::unordered_map<int64_t, Seq> seqs;  // (references to values stay valid across inserts)
  // A batch call stamps each listed request with a fresh epoch: a request already stamped
  // with it is listed twice. No per-call set to build.
  uint64_t epoch = 0;
  std::vector<Seq*> listed;     // the requests of the current batch call, in order
  std::vector<int32_t> scratch;  // page lists of the current call
};

extern "C" {

int pkv_seq_table_create(pkv_allocator* a, int32_t page_size, pkv_seq_table** out) {
  if (!a || !out || page_size <= 0)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_table_create: bad argument");
  *out = new (std::nothrow) pkv_seq_table{a, page_size, {}, 0, {}, {}};
  if (!*out) return pkv::set_error(PKV_EINVAL, "pkv_seq_table_create: out of host memory");
  return PKV_OK;
}

void pkv_seq_table_destroy(pkv_seq_table* t) { delete t; }

}  // extern "C"

namespace {

// A new request on n_shared whole pages; take_refs: one more reference on each (a shared
// prefix), else the caller's references become the request's (pages it was handed, e.g. by a
// prefix-cache lookup).
int seq_add(pkv_seq_table* t, int64_t rid, const int32_t* shared_pages, int32_t n_shared,
            int64_t shared_len, bool take_refs, const char* who) {
  if (!t || n_shared < 0 || (n_shared > 0 && !shared_pages))
    return pkv::set_error(PKV_EINVAL, "%s: bad argument", who);
  if (t->seqs.count(rid))
    return pkv::set_error(PKV_EINVAL, "%s: request %lld exists", who, (long long)rid);
  if (shared_len != (int64_t)n_shared * t->page_size)
    return pkv::set_error(PKV_EINVAL, "%s: a shared prefix must fill whole pages", who);
  for (int32_t i = 0; i < n_shared; ++i)
    if (pkv_refcount(t->alloc, shared_pages[i]) <= 0)
      return pkv::set_error(PKV_EREFCNT, "%s: page %d is not allocated", who, shared_pages[i]);
  if (take_refs && n_shared > 0) {
    const int st = pkv_incref(t->alloc, shared_pages, n_shared);
    if (st != PKV_OK) return st;
  }
  Seq s;
  s.pages.assign(shared_pages, shared_pages + n_shared);
  s.len = shared_len;
  t->seqs.emplace(rid, std::move(s));
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_seq_add(pkv_seq_table* t, int64_t rid, const int32_t* shared_pages, int32_t n_shared,
                int64_t shared_len) {
  return seq_add(t, rid, shared_pages, n_shared, shared_len, true, "pkv_seq_add");
}

int pkv_seq_adopt(pkv_seq_table* t, int64_t rid, const int32_t* pages, int32_t n_pages,
                  int64_t n_tokens) {
  return seq_add(t, rid, pages, n_pages, n_tokens, false, "pkv_seq_adopt");
}

int pkv_seq_fork(pkv_seq_table* t, const int64_t* src_rids, const int64_t* new_rids, int32_t n) {
  if (!t || n < 0 || (n > 0 && (!src_rids || !new_rids)))
    return pkv::set_error(PKV_EINVAL, "pkv_seq_fork: bad argument");
  // all checks first: the forks are made in order only when every one of them can be (a
  // parent may be a request forked earlier in the same list)
  std::unordered_set<int64_t> fresh;
  for (int32_t i = 0; i < n; ++i) {
    if (!t->seqs.count(src_rids[i]) && !fresh.count(src_rids[i]))
      return pkv::set_error(PKV_EINVAL, "pkv_seq_fork: no request %lld", (long long)src_rids[i]);
    if (t->seqs.count(new_rids[i]) || !fresh.insert(new_rids[i]).second)
      return pkv::set_error(PKV_EINVAL, "pkv_seq_fork: request %lld exists",
                            (long long)new_rids[i]);
  }
  for (int32_t i = 0; i < n; ++i) {
    const Seq& src = t->seqs.at(src_rids[i]);
    Seq s;
    s.pages = src.pages;
    s.len = src.len;
    std::vector<int32_t> live;
    live.reserve(s.pages.size());
    for (int32_t p : s.pages)
      if (p >= 0) live.push_back(p);
    if (!live.empty()) {
      const int st = pkv_incref(t->alloc, live.data(), (int32_t)live.size());
      if (st != PKV_OK) return st;  // (pages of a live request are allocated: cannot happen)
    }
    t->seqs.emplace(new_rids[i], std::move(s));
  }
  return PKV_OK;
}

int pkv_seq_free(pkv_seq_table* t, const int64_t* rids, int32_t n) {
  if (!t || n < 0 || (n > 0 && !rids)) return pkv::set_error(PKV_EINVAL, "pkv_seq_free: bad argument");
  const uint64_t ep = ++t->epoch;
  for (int32_t i = 0; i < n; ++i) {
    auto it = t->seqs.find(rids[i]);
    if (it == t->seqs.end() || it->second.mark == ep)
      return pkv::set_error(PKV_EINVAL, "pkv_seq_free: no request %lld (or listed twice)",
                            (long long)rids[i]);
    it->second.mark = ep;
  }
  std::vector<int32_t>& live = t->scratch;
  for (int32_t i = 0; i < n; ++i) {
    auto it = t->seqs.find(rids[i]);
    live.clear();
    for (int32_t p : it->second.pages)
      if (p >= 0) live.push_back(p);
    if (!live.empty()) {
      const int st = pkv_decref(t->alloc, live.data(), (int32_t)live.size());
      if (st != PKV_OK) return st;
    }
    t->seqs.erase(it);
  }
  return PKV_OK;
}

int pkv_seq_reserve(pkv_seq_table* t, const int64_t* rids, const int32_t* counts, int32_t n,
                    int64_t* slots_out, int32_t* copy_src, int32_t* copy_dst, int32_t* n_copies) {
  if (!t || n < 0 || (n > 0 && (!rids || !counts)) || !n_copies)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: bad argument");
  const int32_t P = t->page_size;
  // pass 1: checks, and the pages the batch will take (copies replay the reference counts)
  const uint64_t ep = ++t->epoch;
  std::vector<Seq*>& listed = t->listed;
  listed.clear();
  std::unordered_map<int32_t, int32_t> dropped;  // shared page -> references given up by copies
  int64_t total = 0, need_pages = 0;
  bool any_copy = false;
  for (int32_t i = 0; i < n; ++i) {
    auto it = t->seqs.find(rids[i]);
    if (it == t->seqs.end() || it->second.mark == ep || counts[i] < 0)
      return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: request %lld unknown, listed twice or "
                            "with a negative count", (long long)rids[i]);
    Seq& s = it->second;
    s.mark = ep;
    listed.push_back(&s);
    total += counts[i];
    if (counts[i] > 0) {
      const int64_t lp = s.len / P;
      if (lp < (int64_t)s.pages.size()) {
        const int32_t page = s.pages[lp];
        if (page < 0)
          return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: request %lld writes into a "
                                "released page", (long long)rids[i]);
        const int32_t ref = pkv_refcount(t->alloc, page);
        if (ref <= 0)
          return pkv::set_error(PKV_EREFCNT, "pkv_seq_reserve: page %d is not allocated", page);
        if (ref > 1) {  // shared: copied unless every other holder copied it first
          int32_t& d = dropped[page];
          if (ref - d > 1) {
            ++d;
            ++need_pages;
            any_copy = true;
          }
        }
      }
    }
    const int64_t grow = pages_for(s.len + counts[i], P) - (int64_t)s.pages.size();
    if (grow > 0) need_pages += grow;
  }
  if (total > 0 && !slots_out)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: slots_out is NULL");
  if (any_copy && (!copy_src || !copy_dst))
    return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: copy arrays are NULL");
  if (need_pages > pkv_num_free(t->alloc))
    return pkv::set_error(PKV_ENOPAGES, "pkv_seq_reserve: %lld pages needed, %d free",
                          (long long)need_pages, pkv_num_free(t->alloc));
  // pass 2: copy-on-write, growth and slots (nothing below can fail after pass 1)
  int32_t nc = 0;
  int64_t o = 0;
  for (int32_t i = 0; i < n; ++i) {
    Seq& s = *listed[i];
    const int32_t c = counts[i];
    if (c > 0) {
      int32_t src = -1, dst = -1;
      const int st = pkv_cow_page(t->alloc, s.pages.data(), (int32_t)s.pages.size(), s.len, P,
                                  &src, &dst);
      if (st != PKV_OK) return st;
      if (src >= 0) {
        copy_src[nc] = src;
        copy_dst[nc] = dst;
        ++nc;
      }
    }
    const int64_t grow = pages_for(s.len + c, P) - (int64_t)s.pages.size();
    if (grow > 0) {
      const size_t old = s.pages.size();
      s.pages.resize(old + grow);
      const int st = pkv_alloc(t->alloc, (int32_t)grow, s.pages.data() + old);
      if (st != PKV_OK) return st;
    }
    // slots page by page: page * P + offset, consecutive within a page
    const int64_t end = s.len + c;
    for (int64_t pos = s.len; pos < end;) {
      const int64_t lp = pos / P;
      const int64_t base = (int64_t)s.pages[lp] * P - lp * P;
      const int64_t stop = std::min<int64_t>(end, (lp + 1) * P);
      for (; pos < stop; ++pos) slots_out[o++] = base + pos;
    }
    s.len = end;
  }
  *n_copies = nc;
  return PKV_OK;
}

int pkv_seq_tables(const pkv_seq_table* t, const int64_t* rids, int32_t n, int32_t width,
                   int32_t* block_tables_out, int32_t* context_lens_out) {
  if (!t || n < 0 || (n > 0 && !rids) || width < 0)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_tables: bad argument");
  for (int32_t i = 0; i < n; ++i) {
    auto it = t->seqs.find(rids[i]);
    if (it == t->seqs.end())
      return pkv::set_error(PKV_EINVAL, "pkv_seq_tables: no request %lld", (long long)rids[i]);
    const Seq& s = it->second;
    if (block_tables_out) {
      if ((int64_t)s.pages.size() > width)
        return pkv::set_error(PKV_EINVAL, "pkv_seq_tables: request %lld has %zu pages, the "
                              "table %d columns", (long long)rids[i], s.pages.size(), width);
      int32_t* row = block_tables_out + (int64_t)i * width;
      if (!s.pages.empty()) std::memcpy(row, s.pages.data(), s.pages.size() * sizeof(int32_t));
      std::memset(row + s.pages.size(), 0, (width - s.pages.size()) * sizeof(int32_t));
    }
    if (context_lens_out) {
      if (s.len > INT32_MAX)
        return pkv::set_error(PKV_EINVAL, "pkv_seq_tables: request %lld is longer than int32",
                              (long long)rids[i]);
      context_lens_out[i] = (int32_t)s.len;
    }
  }
  return PKV_OK;
}

int pkv_seq_release_outside_window(pkv_seq_table* t, int64_t rid, int64_t window,
                                   int64_t sink_tokens, int32_t* released) {
  if (!t || window < 0 || sink_tokens < 0)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_release_outside_window: bad argument");
  auto it = t->seqs.find(rid);
  if (it == t->seqs.end())
    return pkv::set_error(PKV_EINVAL, "pkv_seq_release_outside_window: no request %lld",
                          (long long)rid);
  Seq& s = it->second;
  const int32_t P = t->page_size;
  std::vector<int32_t> gone;
  if (window > 0) {
    for (size_t lp = 0; lp < s.pages.size(); ++lp) {
      if (s.pages[lp] < 0) continue;
      const int64_t first = (int64_t)lp * P;
      const int64_t last = std::min<int64_t>(first + P, s.len) - 1;
      // every position of the page is past the sinks, before the window and not the newest
      if (last < s.len - 1 && first >= sink_tokens && last < s.len - window) {
        gone.push_back(s.pages[lp]);
        s.pages[lp] = -1;
      }
    }
  }
  if (!gone.empty()) {
    const int st = pkv_decref(t->alloc, gone.data(), (int32_t)gone.size());
    if (st != PKV_OK) return st;
  }
  if (released) *released = (int32_t)gone.size();
  return PKV_OK;
}

int64_t pkv_seq_len(const pkv_seq_table* t, int64_t rid) {
  if (!t) return -1;
  auto it = t->seqs.find(rid);
  return it == t->seqs.end() ? -1 : it->second.len;
}

int32_t pkv_seq_pages(const pkv_seq_table* t, int64_t rid, int32_t* pages_out, int32_t cap) {
  if (!t) return -1;
  auto it = t->seqs.find(rid);
  if (it == t->seqs.end()) return -1;
  const std::vector<int32_t>& p = it->second.pages;
  if (pages_out && cap > 0)
    std::memcpy(pages_out, p.data(), std::min<size_t>(cap, p.size()) * sizeof(int32_t));
  return (int32_t)p.size();
}

int32_t pkv_seq_count(const pkv_seq_table* t) { return t ? (int32_t)t->seqs.size() : -1; }

int32_t pkv_seq_ids(const pkv_seq_table* t, int64_t* rids_out, int32_t cap) {
  if (!t) return -1;
  int32_t i = 0;
  for (const auto& kv : t->seqs) {
    if (rids_out && i < cap) rids_out[i] = kv.first;
    ++i;
  }
  return i;
}

}  // extern "C"
