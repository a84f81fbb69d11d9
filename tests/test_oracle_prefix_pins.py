"""Pins for the two oracle parts that serve shared prefixes, checked against what the pages fix
and against plain layouts -- never against the oracle itself. CPU only.

* ``oracle.PrefixCacheModel`` -- "KV cache and PagedAttention", section 6 (prefix caching:
  the prefix's KV pages are stored under a key made from its tokens and reused by a later
  request with the same prefix) and pitfall 5 (the tenant belongs in the key); the "KV Cache"
  glossary, prefix caching (the longest common prefix is found and reused). Pages are the
  unit of storage (section 4), so only whole pages are reused. The eviction order is this
  library's reading (the pages name no policy): least recently used first, among entries with
  no cached continuation that no request holds.
* The shared-prefix branch of the C oracle's contiguous decode -- section 4 ("Sharing":
  requests with the same prefix share its pages): attending over a shared prefix followed by
  a request's own tokens must equal attending over the same tokens laid out one after the
  other, and torch's float64 attention over those tokens.

Each pin is a function that raises AssertionError when the implementation it is given is
wrong; the planted-mistake tests hand it a copy of the oracle with one mistake each (a Python
subclass, or the C source with one expression changed and compiled apart) and check that the
pin catches it.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

P = 16


# ---- prefix cache model ---------------------------------------------------------------------

def _prompt(seed, n):
    return np.random.default_rng(seed).integers(0, 1000, n).tolist()


def _pin_whole_pages_and_tenant(model_cls):
    """A 35-token prompt fills two whole pages and part of a third: only the two whole pages
    are stored and reused; another tenant with the same tokens reuses nothing."""
    a = oracle.AllocatorModel(16)
    c = model_cls(a, P)
    toks = _prompt(1, 35)
    pages = a.alloc(3)
    c.insert(7, toks, pages)
    assert len(c.entries) == 2, "a partly filled page was stored"
    assert a.ref[pages[0]] == 2 and a.ref[pages[1]] == 2 and a.ref[pages[2]] == 1
    assert c.lookup(8, toks) == [], "another tenant reused the pages"
    got = c.lookup(7, toks)
    assert got == pages[:2], "the same prompt did not reuse exactly its two whole pages"
    assert a.ref[pages[0]] == 3 and a.ref[pages[1]] == 3 and a.ref[pages[2]] == 1
    # a 47-token prompt with the same first 35 tokens still reuses two pages, a 32-token one too
    assert c.lookup(7, toks + _prompt(2, 12)) == pages[:2]
    assert c.lookup(7, toks[:32]) == pages[:2]
    # 31 tokens hold only one whole page
    assert c.lookup(7, toks[:31]) == pages[:1]


def _pin_longest_prefix(model_cls):
    """The lookup returns the longest run of leading whole pages that match, stopping at the
    first page that differs: a page's keys and values depend on every token before it, so a
    matching later page after a differing one is not a hit."""
    a = oracle.AllocatorModel(32)
    c = model_cls(a, P)
    A = _prompt(3, 4 * P)  # pages A0 A1 A2 A3
    pa = a.alloc(4)
    c.insert(1, A, pa)
    B = A[:2 * P] + _prompt(4, P) + A[3 * P:]  # A0 A1, a different third page, then A3
    assert c.lookup(1, B) == pa[:2]
    Z = _prompt(5, 2 * P)  # Z0 Z1
    pz = a.alloc(2)
    c.insert(1, Z, pz)
    # Z0 followed by A's second page: only Z0 is a hit (A1 was cached after A0, not after Z0)
    assert c.lookup(1, Z[:P] + A[P:2 * P]) == pz[:1]
    # first page differs: nothing, even though pages 1..3 equal A's
    assert c.lookup(1, _prompt(6, P) + A[P:]) == []
    # the whole prompt: all four pages; a lookup capped at two pages returns two
    assert c.lookup(1, A) == pa
    assert c.lookup(1, A, max_pages=2) == pa[:2]


def _pin_eviction(model_cls):
    """Eviction takes least recently used entries first, and only entries that have no cached
    continuation and whose page no request holds (the cache's own reference is the only one)."""
    a = oracle.AllocatorModel(16)
    c = model_cls(a, P)
    A = _prompt(7, 3 * P)
    pa = a.alloc(3)
    c.insert(1, A, pa)  # entries A0 -> A1 -> A2
    B = _prompt(8, P)
    pb = a.alloc(1)
    c.insert(1, B, pb)  # entry B0, used after A's
    a.decref(pa + pb)  # the inserting requests finish: the cache holds the only references
    held = c.lookup(1, A[:P])  # a request holds A0
    assert held == pa[:1] and a.ref[pa[0]] == 2
    # leaves: A2 and B0; A2 is the least recently used of them
    assert c.evict(1) == 1
    assert a.ref[pa[2]] == 0 and a.ref[pb[0]] == 1, "not the least recently used leaf"
    assert a.ref[pa[1]] == 1, "an entry with a cached continuation was evicted"
    # touch A1 (lookup of two pages), so B0 is now older than A1
    got = c.lookup(1, A[:2 * P])
    assert got == pa[:2]
    a.decref(got)
    assert c.evict(1) == 1 and a.ref[pb[0]] == 0 and a.ref[pa[1]] == 1
    assert c.evict(1) == 1 and a.ref[pa[1]] == 0  # A1 is a leaf now
    # A0 is a leaf but a request holds it: nothing can go
    assert c.evict(5) == 0 and a.ref[pa[0]] == 2
    a.decref(held)
    assert c.evict(5) == 1 and a.ref[pa[0]] == 0 and len(c.entries) == 0
    assert a.num_free() == 16


PREFIX_PINS = (_pin_whole_pages_and_tenant, _pin_longest_prefix, _pin_eviction)


@pytest.mark.parametrize("pin", PREFIX_PINS, ids=lambda f: f.__name__)
def test_prefix_cache_model_pins(pin):
    pin(oracle.PrefixCacheModel)


class _NoTenant(oracle.PrefixCacheModel):
    def _key(self, tenant, tokens, i):  # planted: the tenant left out of the key
        return super()._key(0, tokens, i)


class _PartialPage(oracle.PrefixCacheModel):
    def lookup(self, tenant, tokens, max_pages=1 << 20):  # planted: a partial page counts
        return super().lookup(tenant, list(tokens) + [0] * (-len(tokens) % self.P), max_pages)

    def insert(self, tenant, tokens, pages):
        return super().insert(tenant, list(tokens) + [0] * (-len(tokens) % self.P), pages)


class _PageOnlyKey(oracle.PrefixCacheModel):
    def _key(self, tenant, tokens, i):  # planted: page i keyed by its own tokens only
        return (tenant, i > 0, tuple(int(t) for t in tokens[i * self.P:(i + 1) * self.P]))


class _EvictAnything(oracle.PrefixCacheModel):
    def _children(self, key):  # planted: entries with a continuation may go
        return 0


class _EvictHeld(oracle.PrefixCacheModel):
    def evict(self, max_pages):  # planted: pages that requests hold may go as well
        done = 0
        for key in list(self.lru):
            if done >= max_pages:
                break
            if self._children(key) == 0:
                self.a.decref([self.entries.pop(key)])
                self.lru.remove(key)
                done += 1
        return done


class _EvictNewest(oracle.PrefixCacheModel):
    def evict(self, max_pages):  # planted: most recently used first
        self.lru.reverse()
        try:
            return super().evict(max_pages)
        finally:
            self.lru.reverse()


@pytest.mark.parametrize("mutant,pin", [
    (_NoTenant, _pin_whole_pages_and_tenant),
    (_PartialPage, _pin_whole_pages_and_tenant),
    (_PageOnlyKey, _pin_longest_prefix),
    (_EvictAnything, _pin_eviction),
    (_EvictHeld, _pin_eviction),
    (_EvictNewest, _pin_eviction),
], ids=lambda x: x.__name__)
def test_prefix_cache_pins_catch_planted_mistakes(mutant, pin):
    with pytest.raises(AssertionError):
        pin(mutant)


# ---- shared-prefix branch of the contiguous decode ---------------------------------------

def _prefix_case(seed, prefix_len, own, h_q=8, h_kv=2, d=16):
    """Tokens of B requests: a shared prefix [prefix_len, h_kv, d] and own rows. The own rows
    sit between junk rows (one before every request, one at the end) and the prefix array has
    one junk row after it, so an off-by-one read lands on junk and changes the result."""
    rng = np.random.default_rng(seed)
    own = np.asarray(own)
    B = len(own)
    pk = rng.standard_normal((prefix_len + 1, h_kv, d)).astype(np.float32)
    pv = rng.standard_normal((prefix_len + 1, h_kv, d)).astype(np.float32)
    pk[prefix_len] = 50.0
    pv[prefix_len] = -50.0
    rows_k, rows_v, offsets = [], [], []
    n = 0
    own_k, own_v = [], []
    for b in range(B):
        jk = np.full((1, h_kv, d), 40.0, np.float32)
        jv = np.full((1, h_kv, d), 30.0, np.float32)
        k = rng.standard_normal((own[b], h_kv, d)).astype(np.float32)
        v = rng.standard_normal((own[b], h_kv, d)).astype(np.float32)
        rows_k += [jk, k]
        rows_v += [jv, v]
        offsets.append(n + 1)
        n += 1 + own[b]
        own_k.append(k)
        own_v.append(v)
    rows_k.append(np.full((1, h_kv, d), 40.0, np.float32))
    rows_v.append(np.full((1, h_kv, d), 30.0, np.float32))
    q = rng.standard_normal((B, h_q, d)).astype(np.float32)
    return dict(q=q, pk=pk, pv=pv, prefix_len=prefix_len, K=np.concatenate(rows_k),
                V=np.concatenate(rows_v), offsets=np.array(offsets, np.int64),
                lens=(prefix_len + own).astype(np.int32), own_k=own_k, own_v=own_v)


def _pin_prefix_branch(c, scale=0.37, sink=0, window=0, lib_under_test=None):
    """With the prefix: equal, bit for bit, to the same tokens laid out one after the other
    with no prefix, and to torch's float64 attention over them. ``lib_under_test`` (a bound
    build of the C oracle) computes the prefix layout; the plain layout always uses the
    oracle as built."""
    B = len(c["lens"])
    real = oracle.lib()
    oracle._lib = lib_under_test or real
    try:
        got = oracle.contiguous_decode(c["q"], "f32", c["K"], c["V"], "f32", c["offsets"],
                                       c["lens"], scale, prefix_k_raw=c["pk"],
                                       prefix_v_raw=c["pv"], prefix_len=c["prefix_len"],
                                       sink=sink, window=window)
    finally:
        oracle._lib = real
    L = c["prefix_len"]
    flat_k = np.concatenate([np.concatenate([c["pk"][:L], c["own_k"][b]]) for b in range(B)])
    flat_v = np.concatenate([np.concatenate([c["pv"][:L], c["own_v"][b]]) for b in range(B)])
    off = np.concatenate([[0], np.cumsum(c["lens"])[:-1]]).astype(np.int64)
    plain = oracle.contiguous_decode(c["q"], "f32", flat_k, flat_v, "f32", off, c["lens"], scale,
                                     sink=sink, window=window)
    assert np.array_equal(got, plain), "prefix layout differs from the plain layout"
    for b in range(B):
        T = int(c["lens"][b])
        keep = oracle.attended_tokens(T, sink, window)
        k = torch.from_numpy(flat_k[off[b]:off[b] + T][keep].astype(np.float64))
        v = torch.from_numpy(flat_v[off[b]:off[b] + T][keep].astype(np.float64))
        qt = torch.from_numpy(c["q"][b].astype(np.float64))[None, :, None, :]
        o = F.scaled_dot_product_attention(qt, k.transpose(0, 1)[None], v.transpose(0, 1)[None],
                                           scale=scale, enable_gqa=True)[0, :, 0, :].numpy()
        assert np.abs(got[b] - o).max() <= 1e-12, "prefix layout differs from SDPA"


PREFIX_CASES = [
    (21, 32, [3, 16, 20, 1], 0, 0),   # two whole pages shared
    (22, 20, [5, 1, 30], 0, 0),       # a prefix that ends inside a page
    (23, 1, [1, 7], 0, 0),            # a one-token prefix
    (24, 48, [9, 2, 33], 4, 24),      # sinks inside the prefix, window over both parts
    (25, 40, [6, 50], 0, 10),         # window inside the own tokens only
]


@pytest.mark.parametrize("seed,prefix_len,own,sink,window", PREFIX_CASES)
def test_contiguous_decode_prefix_branch_pins(seed, prefix_len, own, sink, window):
    _pin_prefix_branch(_prefix_case(seed, prefix_len, own), sink=sink, window=window)


_PREFIX_MUTANTS = {
    "own row shifted by one": ("((offsets[b] + t - prefix_len) * h_kv + j) * d + i",
                               "((offsets[b] + t - prefix_len - 1) * h_kv + j) * d + i"),
    "prefix one token short": ("if (t < prefix_len) {", "if (t + 1 < prefix_len) {"),
    "prefix one token long": ("if (t < prefix_len) {", "if (t <= prefix_len) {"),
    "V read from the K prefix": ("V[n * d + i] = read_elem(prefix_v, kv_dtype, idx, vs);",
                                 "V[n * d + i] = read_elem(prefix_k, kv_dtype, idx, vs);"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()
    assert src.count(old) == 1, "the expression to change is not unique: %s" % name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", str(path), "-o", str(so), "-lm"], check=True)
    return oracle.bind(ctypes.CDLL(str(so)))


@pytest.mark.parametrize("name", sorted(_PREFIX_MUTANTS))
def test_prefix_branch_pins_catch_planted_mistakes(tmp_path, name):
    mutant = _build_mutant(tmp_path, name, *_PREFIX_MUTANTS[name])
    caught = 0
    for seed, prefix_len, own, sink, window in PREFIX_CASES:
        try:
            _pin_prefix_branch(_prefix_case(seed, prefix_len, own), sink=sink, window=window,
                               lib_under_test=mutant)
        except AssertionError:
            caught += 1
    assert caught > 0, "no pin caught: %s" % name
