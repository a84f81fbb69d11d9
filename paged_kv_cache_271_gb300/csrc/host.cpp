// Host side of the library that needs no GPU: error messages, page accounting, slot mapping
// and the page allocator.
//
// Page allocator ("KV cache and PagedAttention", section 4: pages are uniform and the
// allocator is O(1); requests sharing a prefix share pages, and the "KV Cache" glossary adds
// sharing across sequences for parallel sampling and beam search). A LIFO stack of free page
// ids plus one reference count per page: alloc pops, the last decref pushes back. Every
// request is validated completely before anything changes, so a failed call has no effect.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {

static thread_local char g_msg[512] = "";

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

}  // namespace pkv

struct pkv_allocator {
  int32_t num_pages;
  std::vector<int32_t> stack;  // free ids; back() is handed out next
  std::vector<int32_t> ref;
};

extern "C" {

const char* pkv_last_error(void) { return pkv::g_msg; }

int pkv_version(void) { return 1; }

int pkv_pages_needed(int64_t n_tokens, int32_t page_size, int64_t* pages_out) {
  if (!pages_out || page_size <= 0 || n_tokens < 0)
    return pkv::set_error(PKV_EINVAL, "pkv_pages_needed: bad argument");
  *pages_out = (n_tokens + page_size - 1) / page_size;
  return PKV_OK;
}

int pkv_slot_mapping(const int32_t* block_tables, int32_t max_pages_per_seq,
                     const int32_t* requests, const int64_t* positions, int64_t n,
                     int32_t page_size, int32_t num_pages, int64_t* slots_out) {
  if (n < 0 || (n > 0 && (!block_tables || !positions || !slots_out)) || page_size <= 0 ||
      max_pages_per_seq <= 0 || num_pages <= 0)
    return pkv::set_error(PKV_EINVAL, "pkv_slot_mapping: bad argument");
  for (int64_t i = 0; i < n; ++i) {
    const int64_t p = positions[i];
    if (p < 0) {
      slots_out[i] = -1;
      continue;
    }
    const int64_t r = requests ? requests[i] : i;
    if (r < 0)
      return pkv::set_error(PKV_EINVAL, "pkv_slot_mapping: request %lld < 0", (long long)r);
    const int64_t pi = p / page_size;
    if (pi >= max_pages_per_seq)
      return pkv::set_error(PKV_EINVAL, "pkv_slot_mapping: position %lld beyond the table",
                            (long long)p);
    const int32_t page = block_tables[r * max_pages_per_seq + pi];
    if (page < 0 || page >= num_pages)
      return pkv::set_error(PKV_EINVAL, "pkv_slot_mapping: page id %d out of range", page);
    slots_out[i] = (int64_t)page * page_size + p % page_size;
  }
  return PKV_OK;
}

int pkv_allocator_create(int32_t num_pages, const int32_t* initial_free_order,
                         pkv_allocator** out) {
  if (!out || num_pages <= 0)
    return pkv::set_error(PKV_EINVAL, "pkv_allocator_create: bad argument");
  pkv_allocator* a = new (std::nothrow) pkv_allocator;
  if (!a) return pkv::set_error(PKV_EINVAL, "pkv_allocator_create: out of host memory");
  a->num_pages = num_pages;
  a->ref.assign(num_pages, 0);
  a->stack.resize(num_pages);
  std::vector<char> seen(num_pages, 0);
  for (int32_t k = 0; k < num_pages; ++k) {
    const int32_t id = initial_free_order ? initial_free_order[k] : k;
    if (id < 0 || id >= num_pages || seen[id]) {
      delete a;
      return pkv::set_error(PKV_EINVAL,
                            "pkv_allocator_create: initial order is not a permutation");
    }
    seen[id] = 1;
    a->stack[num_pages - 1 - k] = id;  // first listed = top of the stack
  }
  *out = a;
  return PKV_OK;
}

void pkv_allocator_destroy(pkv_allocator* a) { delete a; }

int pkv_alloc(pkv_allocator* a, int32_t n, int32_t* page_ids_out) {
  if (!a || n < 0 || (n > 0 && !page_ids_out))
    return pkv::set_error(PKV_EINVAL, "pkv_alloc: bad argument");
  if ((size_t)n > a->stack.size())
    return pkv::set_error(PKV_ENOPAGES, "pkv_alloc: %d pages requested, %zu free", n,
                          a->stack.size());
  for (int32_t k = 0; k < n; ++k) {
    const int32_t id = a->stack.back();
    a->stack.pop_back();
    a->ref[id] = 1;
    page_ids_out[k] = id;
  }
  return PKV_OK;
}

static int check_range(const pkv_allocator* a, const int32_t* ids, int32_t n, const char* who) {
  if (!a || n < 0 || (n > 0 && !ids)) return pkv::set_error(PKV_EINVAL, "%s: bad argument", who);
  for (int32_t k = 0; k < n; ++k)
    if (ids[k] < 0 || ids[k] >= a->num_pages)
      return pkv::set_error(PKV_EREFCNT, "%s: page id %d out of range", who, ids[k]);
  return PKV_OK;
}

int pkv_incref(pkv_allocator* a, const int32_t* ids, int32_t n) {
  const int st = check_range(a, ids, n, "pkv_incref");
  if (st != PKV_OK) return st;
  for (int32_t k = 0; k < n; ++k)
    if (a->ref[ids[k]] <= 0)
      return pkv::set_error(PKV_EREFCNT, "pkv_incref: page %d is not allocated", ids[k]);
  for (int32_t k = 0; k < n; ++k) ++a->ref[ids[k]];
  return PKV_OK;
}

int pkv_decref(pkv_allocator* a, const int32_t* ids, int32_t n) {
  const int st = check_range(a, ids, n, "pkv_decref");
  if (st != PKV_OK) return st;
  // Decrement in place; a page reaching 0 goes back on the free stack. If any count would
  // drop below 0 (a free page, or an id listed more often than it is referenced), undo the
  // decrements and pushes made so far, so the call has no effect.
  size_t pushed = 0;
  for (int32_t k = 0; k < n; ++k) {
    const int32_t id = ids[k];
    if (a->ref[id] <= 0) {
      for (int32_t u = k - 1; u >= 0; --u) ++a->ref[ids[u]];
      a->stack.resize(a->stack.size() - pushed);
      return pkv::set_error(PKV_EREFCNT, "pkv_decref: page %d has reference count 0", id);
    }
    if (--a->ref[id] == 0) {
      a->stack.push_back(id);
      ++pushed;
    }
  }
  return PKV_OK;
}

int pkv_cow_page(pkv_allocator* a, int32_t* row, int32_t n, int64_t position,
                 int32_t page_size, int32_t* copy_src, int32_t* copy_dst) {
  if (!a || (n > 0 && !row) || n < 0 || position < 0 || page_size <= 0 || !copy_src || !copy_dst)
    return pkv::set_error(PKV_EINVAL, "pkv_cow_page: bad argument");
  *copy_src = *copy_dst = -1;
  const int64_t lp = position / page_size;
  if (lp >= n) return PKV_OK;  // the write starts a page the request does not have yet
  const int32_t page = row[lp];
  if (page < 0 || page >= a->num_pages || a->ref[page] <= 0)
    return pkv::set_error(PKV_EREFCNT, "pkv_cow_page: page %d is not allocated", page);
  if (a->ref[page] == 1) return PKV_OK;  // private already: write in place
  int32_t fresh = -1;
  const int st = pkv_alloc(a, 1, &fresh);
  if (st != PKV_OK) return st;
  --a->ref[page];  // still referenced by the other sharers (count was > 1)
  row[lp] = fresh;
  *copy_src = page;
  *copy_dst = fresh;
  return PKV_OK;
}

int32_t pkv_num_free(const pkv_allocator* a) { return a ? (int32_t)a->stack.size() : -1; }

int32_t pkv_refcount(const pkv_allocator* a, int32_t id) {
  if (!a || id < 0 || id >= a->num_pages) return -1;
  return a->ref[id];
}

}  // extern "C"
