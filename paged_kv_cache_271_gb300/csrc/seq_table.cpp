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
  // incremental table export: the row of the table's export buffer this request was last
  // written to (-1: none), and the first column changed since
  int64_t exp_row = -1;
  int64_t dirty_from = 0;
  void changed(int64_t col) { dirty_from = std::min(dirty_from, col); }
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
  std::vector<int32_t> ones;     // per-request counts of 1 (pkv_seq_step)
  std::vector<int64_t> slots;    // slots nobody asked for (pkv_seq_step)
  std::vector<Seq*> live_seqs;   // the live requests' entries, looked up once (pkv_seq_step)
  std::vector<Seq*> new_seqs;    // the new requests' entries (pkv_seq_step)
  // incremental table export (pkv_seq_step): the buffer and width it last wrote, and the
  // request whose row each of its rows holds
  mutable const int32_t* inc_buf = nullptr;  // (pkv_seq_tables into it forgets it)
  int32_t inc_width = -1;
  std::vector<int64_t> inc_owner;
};

extern "C" {

int pkv_seq_table_create(pkv_allocator* a, int32_t page_size, pkv_seq_table** out) {
  if (!a || !out || page_size <= 0)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_table_create: bad argument");
  *out = new (std::nothrow)
      pkv_seq_table{a, page_size, {}, 0, {}, {}, {}, {}, {}, {}, nullptr, -1, {}};
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

// Grows the requests seqs[0 .. n) (distinct, counts >= 0: the caller checked) by counts[i]
// tokens each: copy-on-write of a shared, partly filled page about to be written, then the new
// pages and the new tokens' slots; nothing changes unless everything fits (rids: for messages).
int reserve_seqs(pkv_seq_table* t, Seq* const* seqs, const int64_t* rids, const int32_t* counts,
                 int32_t n, int64_t* slots_out, int32_t* copy_src, int32_t* copy_dst,
                 int32_t* n_copies) {
  const int32_t P = t->page_size;
  // pass 1: checks, and the pages the batch will take (copies replay the reference counts)
  std::unordered_map<int32_t, int32_t> dropped;  // shared page -> references given up by copies
  int64_t total = 0, need_pages = 0;
  bool any_copy = false;
  for (int32_t i = 0; i < n; ++i) {
    Seq& s = *seqs[i];
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
    Seq& s = *seqs[i];
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
        s.changed(s.len / P);
      }
    }
    const int64_t grow = pages_for(s.len + c, P) - (int64_t)s.pages.size();
    if (grow > 0) {
      const size_t old = s.pages.size();
      s.changed((int64_t)old);
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
  const uint64_t ep = ++t->epoch;
  std::vector<Seq*>& listed = t->listed;
  listed.clear();
  for (int32_t i = 0; i < n; ++i) {
    auto it = t->seqs.find(rids[i]);
    if (it == t->seqs.end() || it->second.mark == ep || counts[i] < 0)
      return pkv::set_error(PKV_EINVAL, "pkv_seq_reserve: request %lld unknown, listed twice or "
                            "with a negative count", (long long)rids[i]);
    it->second.mark = ep;
    listed.push_back(&it->second);
  }
  return reserve_seqs(t, listed.data(), rids, counts, n, slots_out, copy_src, copy_dst,
                      n_copies);
}

int pkv_seq_tables(const pkv_seq_table* t, const int64_t* rids, int32_t n, int32_t width,
                   int32_t* block_tables_out, int32_t* context_lens_out) {
  if (!t || n < 0 || (n > 0 && !rids) || width < 0)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_tables: bad argument");
  if (block_tables_out && block_tables_out == t->inc_buf) t->inc_buf = nullptr;
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

int pkv_seq_step(pkv_seq_table* t, const int64_t* free_rids, int32_t n_free,
                 const int64_t* new_rids, const int32_t* prompt_counts, int32_t n_new,
                 int64_t* prompt_slots_out, const int64_t* live_rids, int32_t n_live,
                 int64_t* live_slots_out, int32_t width, int32_t* block_tables_out,
                 int32_t* context_lens_out, int32_t incremental, int32_t* copy_src,
                 int32_t* copy_dst, int32_t* n_copies) {
  const char* who = "pkv_seq_step";
  if (!t || n_free < 0 || n_new < 0 || n_live < 0 || width < 0 || !n_copies ||
      (n_free > 0 && !free_rids) || (n_new > 0 && (!new_rids || !prompt_counts)) ||
      (n_live > 0 && !live_rids))
    return pkv::set_error(PKV_EINVAL, "%s: bad argument", who);
  const int32_t P = t->page_size;
  *n_copies = 0;
  // ---- every check first: nothing has changed when one fails ----
  const uint64_t ep_free = ++t->epoch;
  for (int32_t i = 0; i < n_free; ++i) {
    auto it = t->seqs.find(free_rids[i]);
    if (it == t->seqs.end() || it->second.mark == ep_free)
      return pkv::set_error(PKV_EINVAL, "%s: no request %lld to free (or listed twice)", who,
                            (long long)free_rids[i]);
    it->second.mark = ep_free;
  }
  // new requests: distinct, and not live unless freed by this call; value: prompt, listed live
  std::unordered_map<int64_t, std::pair<int32_t, bool>> fresh;
  int64_t prompt_total = 0;
  for (int32_t i = 0; i < n_new; ++i) {
    auto it = t->seqs.find(new_rids[i]);
    if (prompt_counts[i] < 0 || (it != t->seqs.end() && it->second.mark != ep_free) ||
        !fresh.emplace(new_rids[i], std::make_pair(prompt_counts[i], false)).second)
      return pkv::set_error(PKV_EINVAL, "%s: new request %lld exists, is listed twice or has a "
                            "negative prompt", who, (long long)new_rids[i]);
    prompt_total += prompt_counts[i];
  }
  if (prompt_total > 0 && !prompt_slots_out)
    return pkv::set_error(PKV_EINVAL, "%s: prompt_slots_out is NULL", who);
  // live requests: distinct, live after the frees and adds, writable, and fitting the table
  // (each existing one's entry is kept for the reserve and the export below: erasing or adding
  // other entries of the map leaves it in place)
  const uint64_t ep_live = ++t->epoch;
  t->live_seqs.assign(n_live, nullptr);
  for (int32_t i = 0; i < n_live; ++i) {
    int64_t len, pages;
    auto f = fresh.find(live_rids[i]);
    if (f != fresh.end()) {
      if (f->second.second)
        return pkv::set_error(PKV_EINVAL, "%s: request %lld listed twice", who,
                              (long long)live_rids[i]);
      f->second.second = true;
      len = f->second.first;
      pages = pages_for(len, P);
    } else {
      auto it = t->seqs.find(live_rids[i]);
      if (it == t->seqs.end() || it->second.mark == ep_free || it->second.mark == ep_live)
        return pkv::set_error(PKV_EINVAL, "%s: request %lld is not live (or listed twice)", who,
                              (long long)live_rids[i]);
      Seq& s = it->second;
      s.mark = ep_live;
      t->live_seqs[i] = &s;
      len = s.len;
      pages = (int64_t)s.pages.size();
      const int64_t lp = len / P;
      if (lp < pages && s.pages[lp] < 0)
        return pkv::set_error(PKV_EINVAL, "%s: request %lld writes into a released page", who,
                              (long long)live_rids[i]);
      if (lp < pages && (!copy_src || !copy_dst)) {
        // shared once the frees are done: references held by finished requests do not count
        const int32_t page = s.pages[lp];
        int32_t ref = pkv_refcount(t->alloc, page);
        for (int32_t k = 0; k < n_free && ref > 1; ++k) {
          const std::vector<int32_t>& fp = t->seqs.find(free_rids[k])->second.pages;
          ref -= (int32_t)std::count(fp.begin(), fp.end(), page);
        }
        if (ref > 1)
          return pkv::set_error(PKV_EINVAL, "%s: request %lld writes into a shared page and the "
                                "copy arrays are NULL", who, (long long)live_rids[i]);
      }
    }
    if (len + 1 > INT32_MAX && context_lens_out)
      return pkv::set_error(PKV_EINVAL, "%s: request %lld is longer than int32", who,
                            (long long)live_rids[i]);
    if (block_tables_out && std::max(pages, pages_for(len + 1, P)) > width)
      return pkv::set_error(PKV_EINVAL, "%s: request %lld needs more than the table's %d "
                            "columns", who, (long long)live_rids[i], width);
  }
  // ---- the finished requests go (this stands whatever follows) ----
  int st = pkv_seq_free(t, free_rids, n_free);
  if (st != PKV_OK) return st;
  // ---- the new requests and their prompts, then one token for every live request; if the
  // pages run out, the new requests are removed again (their prompt pages go back) ----
  t->new_seqs.resize(n_new);
  for (int32_t i = 0; i < n_new; ++i)
    t->new_seqs[i] = &t->seqs.emplace(new_rids[i], Seq{}).first->second;
  for (int32_t i = 0; i < n_live; ++i)  // the new requests among the live ones
    if (!t->live_seqs[i]) t->live_seqs[i] = &t->seqs.find(live_rids[i])->second;
  auto drop_new = [&]() {
    std::vector<int32_t> live;
    for (int32_t i = 0; i < n_new; ++i) {
      auto it = t->seqs.find(new_rids[i]);
      live.clear();
      for (int32_t p : it->second.pages)
        if (p >= 0) live.push_back(p);
      if (!live.empty()) pkv_decref(t->alloc, live.data(), (int32_t)live.size());
      t->seqs.erase(it);
    }
  };
  int32_t none = 0;
  st = reserve_seqs(t, t->new_seqs.data(), new_rids, prompt_counts, n_new, prompt_slots_out,
                    nullptr, nullptr, &none);
  if (st != PKV_OK) {
    drop_new();
    return st;
  }
  if (n_live > 0) {
    t->ones.assign(n_live, 1);
    int64_t* slots = live_slots_out;
    if (!slots) {
      t->slots.resize(n_live);
      slots = t->slots.data();
    }
    st = reserve_seqs(t, t->live_seqs.data(), live_rids, t->ones.data(), n_live, slots,
                      copy_src, copy_dst, n_copies);
    if (st != PKV_OK) {
      drop_new();
      return st;
    }
  }
  if (!incremental || !block_tables_out) {
    if (block_tables_out) t->inc_buf = nullptr;  // (a full export may reuse that buffer)
    return pkv_seq_tables(t, live_rids, n_live, width, block_tables_out, context_lens_out);
  }
  // incremental: a row that holds this request's row from the last export into this buffer
  // (same width) is written only from the first column changed since; any other row in full
  if (t->inc_buf != block_tables_out || t->inc_width != width) {
    t->inc_buf = block_tables_out;
    t->inc_width = width;
    t->inc_owner.clear();
  }
  if ((int64_t)t->inc_owner.size() < n_live) t->inc_owner.resize(n_live, INT64_MIN);
  for (int32_t i = 0; i < n_live; ++i) {
    Seq& s = *t->live_seqs[i];
    int32_t* row = block_tables_out + (int64_t)i * width;
    const int64_t np = (int64_t)s.pages.size();
    if (t->inc_owner[i] == live_rids[i] && s.exp_row == i) {
      for (int64_t c = s.dirty_from; c < np; ++c) row[c] = s.pages[c];
    } else {
      if (np) std::memcpy(row, s.pages.data(), np * sizeof(int32_t));
      std::memset(row + np, 0, (width - np) * sizeof(int32_t));
      if (s.exp_row >= 0 && s.exp_row < (int64_t)t->inc_owner.size() &&
          t->inc_owner[s.exp_row] == live_rids[i])
        t->inc_owner[s.exp_row] = INT64_MIN;  // that row is stale for this request now
      t->inc_owner[i] = live_rids[i];
      s.exp_row = i;
    }
    s.dirty_from = np;
    if (context_lens_out) context_lens_out[i] = (int32_t)s.len;
  }
  return PKV_OK;
}

int pkv_seq_step_width(const pkv_seq_table* t, const int64_t* new_rids,
                       const int32_t* prompt_counts, int32_t n_new, const int64_t* live_rids,
                       int32_t n_live, int32_t* width_out) {
  if (!t || n_new < 0 || n_live < 0 || (n_new > 0 && (!new_rids || !prompt_counts)) ||
      (n_live > 0 && !live_rids) || !width_out)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_step_width: bad argument");
  const int32_t P = t->page_size;
  int64_t w = 1;
  for (int32_t i = 0; i < n_live; ++i) {
    const int64_t rid = live_rids[i];
    int32_t k = 0;
    while (k < n_new && new_rids[k] != rid) ++k;
    if (k < n_new) {
      if (prompt_counts[k] < 0)
        return pkv::set_error(PKV_EINVAL, "pkv_seq_step_width: negative prompt");
      w = std::max(w, pages_for((int64_t)prompt_counts[k] + 1, P));
      continue;
    }
    auto it = t->seqs.find(rid);
    if (it == t->seqs.end())
      return pkv::set_error(PKV_EINVAL, "pkv_seq_step_width: no request %lld", (long long)rid);
    w = std::max(w, std::max((int64_t)it->second.pages.size(), pages_for(it->second.len + 1, P)));
  }
  if (w > INT32_MAX) return pkv::set_error(PKV_EINVAL, "pkv_seq_step_width: row too wide");
  *width_out = (int32_t)w;
  return PKV_OK;
}

int pkv_seq_add_cached_prefix(pkv_seq_table* t, int64_t rid, pkv_prefix_cache* c, int64_t tenant,
                              const int32_t* tokens, int64_t n_tokens, int64_t* cached_tokens) {
  if (!t || !c || n_tokens < 0 || (n_tokens > 0 && !tokens) || !cached_tokens)
    return pkv::set_error(PKV_EINVAL, "pkv_seq_add_cached_prefix: bad argument");
  if (t->seqs.count(rid))
    return pkv::set_error(PKV_EINVAL, "pkv_seq_add_cached_prefix: request %lld exists",
                          (long long)rid);
  const int64_t whole = n_tokens / t->page_size;
  std::vector<int32_t>& pages = t->scratch;
  pages.assign((size_t)std::max<int64_t>(whole, 1), -1);
  int32_t n = 0;
  int st = pkv_prefix_lookup(c, tenant, tokens, n_tokens, pages.data(),
                             (int32_t)std::min<int64_t>(whole, INT32_MAX), &n);
  if (st != PKV_OK) return st;
  st = seq_add(t, rid, pages.data(), n, (int64_t)n * t->page_size, false,
               "pkv_seq_add_cached_prefix");
  if (st != PKV_OK) {
    if (n > 0) pkv_decref(t->alloc, pages.data(), n);  // hand the lookup's references back
    return st;
  }
  *cached_tokens = (int64_t)n * t->page_size;
  return PKV_OK;
}

int pkv_prefix_insert_request(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens,
                              int64_t n_tokens, const pkv_seq_table* t, int64_t rid) {
  if (!c || !t || n_tokens < 0 || (n_tokens > 0 && !tokens))
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_insert_request: bad argument");
  auto it = t->seqs.find(rid);
  if (it == t->seqs.end())
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_insert_request: no request %lld",
                          (long long)rid);
  const Seq& s = it->second;
  const int64_t n = std::min(n_tokens, s.len);  // tokens both written and given
  const int64_t full = std::min<int64_t>(n / t->page_size, (int64_t)s.pages.size());
  if (full == 0) return PKV_OK;
  return pkv_prefix_insert(c, tenant, tokens, full * t->page_size, s.pages.data(),
                           (int32_t)full);
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
        s.changed((int64_t)lp);
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
