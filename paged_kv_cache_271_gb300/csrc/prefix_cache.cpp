// Prefix cache: reuse the KV pages of a prompt prefix seen before ("KV cache and
// PagedAttention", section 6: hash the prefix tokens, store its pages under that hash, reuse
// them for the next request with the same prefix; the "KV Cache" glossary: a radix tree finds
// the longest common prefix; pitfall 5: the tenant / user id must be part of the key).
//
// Every full page of a cached prompt is an entry keyed by a chained hash
//   h_0 = H(tenant, tokens[0:P]),  h_i = H(h_{i-1}, tokens[iP:(i+1)P])
// so an entry names the whole prefix up to and including its page, and a lookup walks the
// chain page by page: the longest cached prefix in whole pages, which is what a radix tree over
// page-sized token blocks returns. Each entry also keeps its tenant, parent hash and tokens and
// a lookup compares them, so a hash collision can never hand one prompt's (or tenant's) pages
// to another. The cache holds one reference on every page it lists (pkv_incref); a lookup
// gives the caller one more reference per matched page. Eviction drops least recently used
// entries that end a cached chain (no cached continuation) and whose page nobody else
// references, in passes over the LRU order until enough are gone or none qualifies.
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "pkv_host.h"

namespace {

uint64_t mix64(uint64_t x) {  // splitmix64 finaliser
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

uint64_t chain_hash(uint64_t parent, int64_t tenant, const int32_t* tokens, int32_t n) {
  uint64_t h = mix64(parent ^ mix64((uint64_t)tenant + 0x5151u));
  for (int32_t i = 0; i < n; ++i) h = mix64(h ^ (uint32_t)tokens[i]);
  return h;
}

struct Entry {
  uint64_t hash;
  uint64_t parent;  // 0 for the first page of a prompt
  int64_t tenant;
  std::vector<int32_t> tokens;
  int32_t page;
  int32_t children = 0;  // cached entries whose parent is this one
  std::list<uint64_t>::iterator lru;
};

}  // namespace

struct pkv_prefix_cache {
  pkv_allocator* alloc;
  int32_t page_size;
  std::unordered_map<uint64_t, Entry> map;
  std::list<uint64_t> lru;  // front = least recently used
};

namespace {

Entry* find(pkv_prefix_cache* c, uint64_t parent, int64_t tenant, const int32_t* tokens) {
  const uint64_t h = chain_hash(parent, tenant, tokens, c->page_size);
  auto it = c->map.find(h);
  if (it == c->map.end()) return nullptr;
  Entry& e = it->second;
  if (e.parent != parent || e.tenant != tenant ||
      std::memcmp(e.tokens.data(), tokens, sizeof(int32_t) * c->page_size) != 0)
    return nullptr;  // a collision, not a match
  return &e;
}

void touch(pkv_prefix_cache* c, Entry& e) { c->lru.splice(c->lru.end(), c->lru, e.lru); }

}  // namespace

extern "C" {

int pkv_prefix_cache_create(pkv_allocator* a, int32_t page_size, pkv_prefix_cache** out) {
  if (!a || page_size <= 0 || !out)
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_cache_create: bad argument");
  pkv_prefix_cache* c = new (std::nothrow) pkv_prefix_cache;
  if (!c) return pkv::set_error(PKV_EINVAL, "pkv_prefix_cache_create: out of host memory");
  c->alloc = a;
  c->page_size = page_size;
  *out = c;
  return PKV_OK;
}

void pkv_prefix_cache_destroy(pkv_prefix_cache* c) {
  if (!c) return;
  for (auto& kv : c->map) pkv_decref(c->alloc, &kv.second.page, 1);
  delete c;
}

int pkv_prefix_lookup(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens, int64_t n,
                      int32_t* pages_out, int32_t max_pages, int32_t* n_pages_out) {
  if (!c || n < 0 || (n > 0 && !tokens) || max_pages < 0 || (max_pages > 0 && !pages_out) ||
      !n_pages_out)
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_lookup: bad argument");
  const int32_t P = c->page_size;
  std::vector<Entry*> hit;
  uint64_t parent = 0;
  for (int64_t i = 0; (i + 1) * P <= n && (int32_t)hit.size() < max_pages; ++i) {
    Entry* e = find(c, parent, tenant, tokens + i * P);
    if (!e) break;
    hit.push_back(e);
    parent = e->hash;
  }
  std::vector<int32_t> ids;
  for (Entry* e : hit) ids.push_back(e->page);
  if (!ids.empty()) {
    const int st = pkv_incref(c->alloc, ids.data(), (int32_t)ids.size());
    if (st != PKV_OK) return st;
  }
  for (size_t k = 0; k < hit.size(); ++k) {
    pages_out[k] = ids[k];
    touch(c, *hit[k]);
  }
  *n_pages_out = (int32_t)hit.size();
  return PKV_OK;
}

int pkv_prefix_insert(pkv_prefix_cache* c, int64_t tenant, const int32_t* tokens, int64_t n,
                      const int32_t* pages, int32_t n_pages) {
  if (!c || n < 0 || (n > 0 && !tokens) || n_pages < 0 || (n_pages > 0 && !pages))
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_insert: bad argument");
  const int32_t P = c->page_size;
  const int64_t full = n / P < n_pages ? n / P : n_pages;
  for (int64_t i = 0; i < full; ++i)
    if (pkv_refcount(c->alloc, pages[i]) <= 0)
      return pkv::set_error(PKV_EREFCNT, "pkv_prefix_insert: page %d is not allocated", pages[i]);
  uint64_t parent = 0;
  Entry* prev = nullptr;
  for (int64_t i = 0; i < full; ++i) {
    const int32_t* blk = tokens + i * P;
    Entry* e = find(c, parent, tenant, blk);
    if (!e) {
      const uint64_t h = chain_hash(parent, tenant, blk, P);
      if (c->map.count(h)) break;  // a colliding entry owns this hash: stop caching here
      int32_t pid = pages[i];
      const int st = pkv_incref(c->alloc, &pid, 1);
      if (st != PKV_OK) return st;
      Entry ne;
      ne.hash = h;
      ne.parent = parent;
      ne.tenant = tenant;
      ne.tokens.assign(blk, blk + P);
      ne.page = pid;
      ne.lru = c->lru.insert(c->lru.end(), h);
      e = &c->map.emplace(h, std::move(ne)).first->second;
      if (prev) ++prev->children;
    } else {
      touch(c, *e);
    }
    parent = e->hash;
    prev = e;
  }
  return PKV_OK;
}

int pkv_prefix_evict(pkv_prefix_cache* c, int32_t max_pages, int32_t* n_evicted) {
  if (!c || max_pages < 0 || !n_evicted)
    return pkv::set_error(PKV_EINVAL, "pkv_prefix_evict: bad argument");
  int32_t done = 0;
  bool progress = true;
  while (done < max_pages && progress) {
    progress = false;
    for (auto it = c->lru.begin(); it != c->lru.end() && done < max_pages;) {
      auto me = c->map.find(*it);
      Entry& e = me->second;
      // only leaves (no cached continuation) whose page nobody but the cache holds
      if (e.children == 0 && pkv_refcount(c->alloc, e.page) == 1) {
        if (e.parent) {
          auto pe = c->map.find(e.parent);
          if (pe != c->map.end()) --pe->second.children;
        }
        pkv_decref(c->alloc, &e.page, 1);
        it = c->lru.erase(it);
        c->map.erase(me);
        ++done;
        progress = true;
      } else {
        ++it;
      }
    }
  }
  *n_evicted = done;
  return PKV_OK;
}

int32_t pkv_prefix_size(const pkv_prefix_cache* c) { return c ? (int32_t)c->map.size() : -1; }

}  // extern "C"
