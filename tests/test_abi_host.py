"""The C-ABI library without a GPU: it loads, exports every declared entry point, and its host
logic (page accounting, slot mapping, allocator, argument checks) agrees with the oracle."""
import ctypes
import os
import re
import time

import numpy as np
import pytest

import oracle
import paged_kv_cache_271_gb300 as pkv
from paged_kv_cache_271_gb300.cache import PagedKVCache

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_271_gb300 import build
    build.build()


def _declared():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_entry_point():
    names = _declared()
    assert len(names) >= 20
    L = ctypes.CDLL(pkv.library_path)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert pkv.lib().pkv_version() == 1


@pytest.mark.parametrize("P", [1, 16, 32])
def test_pages_needed_matches_oracle(P):
    for n in range(0, 300):
        assert pkv.pages_needed(n, P) == oracle.pages_needed(n, P)


def test_slot_mapping_matches_oracle_bit_exact():
    rng = np.random.default_rng(0)
    for _ in range(20):
        B, W, num_pages, P = rng.integers(1, 9), rng.integers(1, 12), 200, 16
        bt = rng.integers(0, num_pages, (B, W)).astype(np.int32)
        n = 100
        req = rng.integers(0, B, n).astype(np.int32)
        pos = rng.integers(-2, W * P, n).astype(np.int64)
        got = pkv.slot_mapping(bt, pos, num_pages, requests=req, page_size=P)
        ref = oracle.slot_mapping(bt, pos, P, requests=req)
        np.testing.assert_array_equal(got, ref)


def test_slot_mapping_rejects_bad_tables():
    bt = np.array([[3, 4]], dtype=np.int32)
    with pytest.raises(pkv.PkvError):
        pkv.slot_mapping(bt, [32], 10)  # position beyond the table width
    with pytest.raises(pkv.PkvError):
        pkv.slot_mapping(np.array([[11]], dtype=np.int32), [0], 10)  # page id outside the pool


def test_allocator_fuzz_against_model():
    rng = np.random.default_rng(1)
    for trial in range(5):
        n = int(rng.integers(1, 64))
        order = rng.permutation(n)
        a = pkv.PageAllocator(n, order)
        m = oracle.AllocatorModel(n, order)
        live = []
        for _ in range(400):
            op = rng.integers(0, 3)
            if op == 0:
                k = int(rng.integers(0, 8))
                try:
                    ref = m.alloc(k)
                except MemoryError:
                    with pytest.raises(pkv.PkvError) as e:
                        a.alloc(k)
                    assert e.value.code == -5
                    continue
                got = a.alloc(k)
                assert list(got) == ref
                live.extend(ref)
            elif op == 1 and live:
                ids = list(rng.choice(live, size=int(rng.integers(1, 4))))
                m.incref(ids)
                a.incref(ids)
                live.extend(ids)
            else:
                ids = list(rng.choice(np.arange(n), size=int(rng.integers(1, 3))))
                try:
                    m.decref(ids)
                except (ValueError, IndexError):
                    with pytest.raises(pkv.PkvError) as e:
                        a.decref(ids)
                    assert e.value.code == -6
                    continue
                a.decref(ids)
                for i in ids:
                    live.remove(i)
            assert a.num_free() == m.num_free()
            for p in range(n):
                assert a.refcount(p) == m.ref[p]
            assert a.num_free() + sum(1 for p in range(n) if a.refcount(p) > 0) == n


def test_allocator_is_constant_time_per_page():
    n = 1 << 20
    a = pkv.PageAllocator(n)
    t0 = time.perf_counter()
    ids = a.alloc(n)
    a.decref(ids)
    t_big = time.perf_counter() - t0
    assert a.num_free() == n
    # one million pages allocated and freed well inside a second: no per-page scans
    assert t_big < 1.0, t_big
    with pytest.raises(pkv.PkvError):
        a.alloc(n + 1)
    assert a.num_free() == n


def test_allocator_rejects_bad_initial_order():
    with pytest.raises(pkv.PkvError):
        pkv.PageAllocator(4, [0, 1, 1, 3])


def _desc(**kw):
    d = dict(num_pages=8, page_size=16, num_kv_heads=2, head_dim=64, cache_dtype=pkv.F32)
    d.update(kw)
    return pkv._Desc(d["num_pages"], d["page_size"], d["num_kv_heads"], d["head_dim"],
                     d["cache_dtype"])


def _decode_status(desc, dtype_q=pkv.F32, h_q=4, ws=None, wsb=0):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails its host checks
    return pkv.lib().pkv_paged_decode_attention(fake, dtype_q, 2, h_q, fake, fake,
                                                ctypes.byref(desc), fake, 600, fake, 0.125,
                                                None, None, fake, ws, wsb, None)


def test_decode_argument_errors_are_caught_on_the_host():
    assert _decode_status(_desc(page_size=8)) == -1
    assert _decode_status(_desc(head_dim=96)) == -2
    assert _decode_status(_desc(), h_q=6) == -2  # group 3
    assert _decode_status(_desc(), dtype_q=pkv.BF16) == -3  # bf16 q on an fp32 cache
    assert _decode_status(_desc(cache_dtype=pkv.FP8_E4M3)) == -1  # FP8 without scales
    assert _decode_status(_desc(cache_dtype=7)) == -3
    # 600 pages per row with batch 2 needs the split, and no workspace was given
    assert _decode_status(_desc()) == -1
    assert "workspace" in pkv.lib().pkv_last_error().decode()


def test_append_argument_errors_are_caught_on_the_host():
    fake = ctypes.c_void_p(1 << 20)
    L = pkv.lib()
    d = _desc(cache_dtype=pkv.BF16)
    assert L.pkv_kv_append(fake, fake, pkv.F32, 4, fake, fake, fake, ctypes.byref(d), None, None,
                           None) == -3
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert L.pkv_kv_append(odd, fake, pkv.BF16, 4, fake, fake, fake, ctypes.byref(d), None,
                           None, None) == -4
    assert L.pkv_kv_append(fake, fake, pkv.BF16, 0, fake, fake, fake, ctypes.byref(d), None,
                           None, None) == 0  # nothing to do


def test_workspace_size_and_chunk_policy():
    pkv.decode_set_chunk_pages(0)
    # Llama-3-8B-shaped batch 64: chunks of at most 32 pages over a 256-page table
    assert pkv.decode_chunk_pages(64, 8, 256) == 32
    # Llama-3-70B-shaped long contexts (4 x 8 units over 8192 pages): 64-page chunks
    assert pkv.decode_chunk_pages(4, 8, 8192) == 64
    rows = 64 * 32 * 8
    # partial values, partial (max, sum); the balanced split's values and (max, sum) for
    # 64 * 8 + 2432 partial slots per query head; then one counter per (request, kv head)
    flat = (64 * 8 + 2432) * 4
    # (and the requests' page offsets, 65 ints in a 256-byte aligned region)
    assert pkv.decode_workspace_size(64, 32, 8, 128, 256) == (rows * 128 * 4 + rows * 2 * 4 +
                                                              flat * 128 * 4 + flat * 2 * 4 +
                                                              512 + 256 * 8)
    pkv.decode_set_chunk_pages(32)  # a chosen chunk size: chunks only, no balanced region
    try:
        assert pkv.decode_workspace_size(64, 32, 8, 128, 256) == (rows * 128 * 4 + rows * 2 * 4 +
                                                                  256 * 8)
    finally:
        pkv.decode_set_chunk_pages(0)
    # the balanced split keeps the requests' page offsets in shared memory, for at most 2048
    # requests: a larger batch has no balanced region (the size of the same 64-page chunks
    # chosen by hand), a batch of 2048 still has one
    assert pkv.decode_chunk_pages(2049, 8, 69) == 64
    auto_2049 = pkv.decode_workspace_size(2049, 32, 8, 128, 69)
    auto_2048 = pkv.decode_workspace_size(2048, 32, 8, 128, 69)
    pkv.decode_set_chunk_pages(64)
    try:
        assert auto_2049 == pkv.decode_workspace_size(2049, 32, 8, 128, 69)
        assert auto_2048 > pkv.decode_workspace_size(2048, 32, 8, 128, 69)
    finally:
        pkv.decode_set_chunk_pages(0)
    # everything fits one chunk: no workspace
    assert pkv.decode_workspace_size(2, 4, 2, 64, 3) == 0
    pkv.decode_set_chunk_pages(2)
    try:
        assert pkv.decode_chunk_pages(2, 2, 3) == 2
        assert pkv.decode_workspace_size(2, 4, 2, 64, 3) > 0
    finally:
        pkv.decode_set_chunk_pages(0)
    with pytest.raises(pkv.PkvError):
        pkv.decode_set_chunk_pages(-1)


def test_cache_bookkeeping_matches_oracle_without_gpu():
    import torch
    order = np.random.default_rng(3).permutation(40)
    c = PagedKVCache(40, 2, 64, torch.float32, device="cpu", initial_free_order=order)
    m = oracle.AllocatorModel(40, order)
    c.add_request(0)
    slots = c.reserve([0], [17])
    pages = m.alloc(2)
    assert c.pages[0] == pages
    np.testing.assert_array_equal(
        slots, oracle.slot_mapping(np.array([pages]), np.arange(17), requests=np.zeros(17, int)))
    # a prefix of two full pages shared by two more requests
    c.add_request(1)
    c.reserve([1], [32])
    shared = list(c.pages[1])
    c.add_request(2, shared_pages=shared, shared_len=32)
    c.add_request(3, shared_pages=shared, shared_len=32)
    assert [c.allocator.refcount(p) for p in shared] == [3, 3]
    s2 = c.reserve([2, 3], [1, 1])
    assert s2[0] // 16 not in shared and s2[1] // 16 not in shared and s2[0] != s2[1]
    c.free_request(1)
    c.free_request(2)
    assert [c.allocator.refcount(p) for p in shared] == [1, 1]
    c.free_request(3)
    c.free_request(0)
    assert c.allocator.num_free() == 40


def test_release_outside_window_bookkeeping():
    import torch
    c = PagedKVCache(20, 2, 64, torch.float32, device="cpu")
    c.add_request(0)
    c.reserve([0], [100])  # 7 pages: positions 0..99
    pages = list(c.pages[0])
    # window of the last 20 positions (80..99) plus 4 sinks (0..3): pages 1..4 hold none
    assert c.release_outside_window(0, 20, 4) == 4
    assert c.pages[0] == [pages[0], -1, -1, -1, -1, pages[5], pages[6]]
    assert c.allocator.num_free() == 20 - 3
    assert c.release_outside_window(0, 20, 4) == 0  # idempotent
    assert c.release_outside_window(0, 0) == 0  # no window: nothing to release
    bt = c.block_table_array([0])
    assert list(bt[0, :7]) == c.pages[0]
    c.reserve([0], [20])  # the window moves on; new pages still map by position
    assert len(c.pages[0]) == 8
    c.free_request(0)
    assert c.allocator.num_free() == 20


def test_copy_on_write_page_logic():
    a = pkv.PageAllocator(10)
    row = list(a.alloc(3))  # positions 0..47 on three private pages
    assert a.cow_page(row, 40) is None  # private: write in place
    a.incref(row)  # a fork shares all three
    shared = list(row)
    pair = a.cow_page(row, 40)  # write into the shared, partly filled third page
    assert pair == (shared[2], row[2]) and row[2] != shared[2]
    assert a.refcount(shared[2]) == 1 and a.refcount(row[2]) == 1
    assert row[:2] == shared[:2] and a.refcount(shared[0]) == 2
    assert a.cow_page(row, 48) is None  # a new page, nothing to copy
    assert a.num_free() + sum(1 for p in range(10) if a.refcount(p) > 0) == 10
    small = pkv.PageAllocator(1)
    r = list(small.alloc(1))
    small.incref(r)
    with pytest.raises(pkv.PkvError):
        small.cow_page(r, 3)  # no free page for the copy: nothing changes
    assert small.refcount(r[0]) == 2


def test_prefix_cache_against_model():
    rng = np.random.default_rng(7)
    P = 16
    for trial in range(3):
        n = 64
        a, am = pkv.PageAllocator(n), oracle.AllocatorModel(n)
        c, cm = pkv.PrefixCache(a, P), oracle.PrefixCacheModel(am, P)
        vocab = [rng.integers(0, 50, 80).tolist() for _ in range(4)]  # a few shared prompts
        held = []  # (pages) referenced by "requests"
        for _ in range(150):
            op = rng.integers(0, 4)
            tenant = int(rng.integers(0, 2))
            base = vocab[int(rng.integers(0, len(vocab)))]
            cut = int(rng.integers(0, len(base) + 1))
            tokens = base[:cut] + rng.integers(0, 50, int(rng.integers(0, 20))).tolist()
            if op <= 1:  # a request arrives: reuse the cached prefix, allocate the rest, cache it
                got, ref = c.lookup(tenant, tokens), cm.lookup(tenant, tokens)
                assert got == ref
                need = -(-len(tokens) // P) - len(got)
                if need > am.num_free():
                    for p in got:
                        a.decref([p]), am.decref([p])
                    continue
                fresh, fresh_m = list(a.alloc(need)), am.alloc(need)
                assert fresh == fresh_m
                pages = got + fresh
                c.insert(tenant, tokens, pages)
                cm.insert(tenant, tokens, pages)
                held.append(pages)
            elif op == 2 and held:  # a request finishes
                pages = held.pop(int(rng.integers(0, len(held))))
                a.decref(pages), am.decref(pages)
            else:
                k = int(rng.integers(0, 8))
                assert c.evict(k) == cm.evict(k)
            assert c.size() == len(cm.entries)
            assert a.num_free() == am.num_free()
            for p in range(n):
                assert a.refcount(p) == am.ref[p]
        for pages in held:
            a.decref(pages)
        del c
        assert a.num_free() == n  # destroying the cache releases its references


def test_prefix_cache_separates_tenants():
    a = pkv.PageAllocator(8)
    c = pkv.PrefixCache(a, 16)
    toks = list(range(40))
    pages = list(a.alloc(3))
    c.insert(tenant=1, tokens=toks, pages=pages)
    assert c.size() == 2  # two full pages
    assert c.lookup(tenant=2, tokens=toks) == []  # another tenant: no reuse
    hit = c.lookup(tenant=1, tokens=toks[:35] + [99])
    assert hit == pages[:2] and a.refcount(pages[0]) == 3
    assert c.lookup(tenant=1, tokens=[7] + toks[1:]) == []  # first page differs


def _groups_model(bt, cl, min_members=2, min_prefix=1):
    """Plain restatement of the grouping rule: bucket by first page in batch order, share the
    longest common run of leading page ids, cut to the full pages before position ctx - 1."""
    B = bt.shape[0]
    cap = [min(max(int(c) - 1, 0) // 16, bt.shape[1]) for c in cl]
    buckets = {}
    for b in range(B):
        if cap[b] >= min_prefix:
            buckets.setdefault(int(bt[b, 0]), []).append(b)
    out = []
    for mem in buckets.values():  # dicts keep insertion (first appearance) order
        if len(mem) < min_members:
            continue
        n = min(cap[b] for b in mem)
        for b in mem[1:]:
            k = 0
            while k < n and bt[b, k] == bt[mem[0], k]:
                k += 1
            n = k
        if n >= min_prefix:
            out.append((mem, n))
    return out


def test_cascade_groups_against_model():
    rng = np.random.default_rng(3)
    for trial in range(200):
        B, W = int(rng.integers(1, 24)), int(rng.integers(1, 12))
        prompts = rng.integers(0, 6, (4, W))  # a few shared page runs
        bt = np.empty((B, W), np.int32)
        for b in range(B):
            p = prompts[rng.integers(0, 4)].copy()
            cut = int(rng.integers(0, W + 1))
            p[cut:] = rng.integers(100, 1000, W - cut)
            bt[b] = p
        cl = rng.integers(0, 16 * W + 1, B).astype(np.int32)
        mm, mp = int(rng.integers(1, 4)), int(rng.integers(0, 3))
        g = pkv.cascade_groups(bt, cl, min_members=mm, min_prefix_pages=mp)
        ref = _groups_model(bt, cl, max(mm, 2), max(mp, 1))
        assert g.n_groups == len(ref)
        got = [(g.group_members[g.group_offsets[i]:g.group_offsets[i + 1]].tolist(),
                int(g.prefix_pages[i])) for i in range(g.n_groups)]
        assert got == ref
        of = np.full(B, -1)
        for i, (mem, _) in enumerate(ref):
            of[mem] = i
        assert np.array_equal(g.group_of, of)
        assert g.max_members == max([len(m) for m, _ in ref], default=0)
        assert g.max_prefix_pages == max([n for _, n in ref], default=0)
        pre = {b: n for mem, n in ref for b in mem}
        own = [-(-min(max(int(cl[b]), 0), 16 * W) // 16) - pre.get(b, 0) for b in range(B)]
        assert g.max_own_pages == max(own, default=0)
        assert g.own_start.tolist() == [pre.get(b, 0) for b in range(B)]
        # each group's shared page ids: its members' common first table entries, -1 padded
        if g.n_groups:
            ids = g.prefix_page_ids.reshape(g.n_groups, g.max_prefix_pages)
            for i, (mem, n) in enumerate(ref):
                assert all(bt[b, :n].tolist() == ids[i, :n].tolist() for b in mem)
                assert (ids[i, n:] == -1).all()
        else:
            assert g.prefix_page_ids is None
    # malformed groups are refused before any table row is read
    L = pkv.lib()
    bt = np.zeros((2, 4), np.int32)
    ids = np.zeros(8, np.int32)
    for members, offs in (([5], [0, 1]), ([0], [0, 0]), ([-1], [0, 1])):
        m = np.array(members, np.int32)
        o = np.array(offs, np.int32)
        pp = np.array([2], np.int32)
        assert L.pkv_cascade_prefix_page_ids(bt.ctypes.data, 2, 4, pp.ctypes.data, o.ctypes.data,
                                             m.ctypes.data, 1, 2, ids.ctypes.data) == -1


def test_cascade_argument_errors_are_caught_on_the_host():
    L = pkv.lib()
    fake = ctypes.c_void_p(1 << 20)
    d = _desc(cache_dtype=pkv.BF16)
    d.head_dim = 128
    good = pkv._CascadeDesc(fake, fake, fake, fake, 1, 2, 3)

    def call(gd, dtype_q=pkv.BF16, desc=d, maxp=600):
        return L.pkv_cascade_decode_attention(fake, dtype_q, 2, 8, fake, fake, ctypes.byref(desc),
                                              fake, maxp, fake, 0.1, ctypes.byref(gd), fake, None,
                                              0, None)
    assert call(pkv._CascadeDesc(None, fake, fake, fake, 1, 2, 3)) == -1  # null array
    assert call(pkv._CascadeDesc(fake, fake, fake, fake, 1, 3, 3)) == -1  # members > batch
    assert call(pkv._CascadeDesc(fake, fake, fake, fake, 1, 2, 601)) == -1  # prefix > table
    f32 = _desc(cache_dtype=pkv.F32)
    f32.head_dim = 128
    assert call(good, dtype_q=pkv.F32, desc=f32) == -3  # the prefix pass is bf16 only
    assert call(good) == -1  # needs a workspace
    assert "workspace" in L.pkv_last_error().decode()
    g = pkv.CascadeGroups(np.zeros(2, np.int32), np.array([3], np.int32), np.array([0, 2], np.int32),
                          np.array([0, 1], np.int32), 2, 3)
    plain = pkv.decode_workspace_size(2, 8, 4, 128, 600)
    # more partial slots than the plain decode's chunks (whose layout, under a chosen chunk
    # size, has no balanced-split region)
    pkv.decode_set_chunk_pages(pkv.decode_chunk_pages(2, 4, 600))
    try:
        chunks_only = pkv.decode_workspace_size(2, 8, 4, 128, 600)
    finally:
        pkv.decode_set_chunk_pages(0)
    assert chunks_only < plain
    assert pkv.cascade_workspace_size(2, 8, 4, 128, 600, g) > chunks_only
    none = pkv.CascadeGroups(np.full(2, -1, np.int32), np.zeros(0, np.int32), np.zeros(1, np.int32),
                             np.zeros(0, np.int32), 0, 0)
    assert pkv.cascade_workspace_size(2, 8, 4, 128, 600, none) == plain
    # tuning switches reject values outside their range and keep their setting
    assert L.pkv_cascade_set_overlap(3) == -1
    assert L.pkv_cascade_set_prefix_kernel(3) == -1
    assert L.pkv_decode_set_warp_per_request(-1) == -1
    pkv.cascade_set_overlap(2)


def test_packed_step_layout():
    L = pkv.lib()
    offs = (ctypes.c_size_t * 5)()
    total = ctypes.c_size_t(0)
    assert L.pkv_packed_step_layout(64, 32, 8, 128, 256, pkv.BF16, pkv.BF16, offs,
                                    ctypes.byref(total)) == 0
    sizes = [64 * 32 * 128 * 2, 64 * 8 * 128 * 2, 64 * 8 * 128 * 2, 64 * 256 * 4, 64 * 4]
    expect, o = [], 0
    for n in sizes:
        expect.append(o)
        o += (n + 255) // 256 * 256
    assert list(offs) == expect and total.value == o
    assert L.pkv_packed_step_layout(1, 4, 2, 64, 3, pkv.FP8_E4M3, pkv.BF16, offs,
                                    ctypes.byref(total)) == -3  # q must be F32 or BF16


def test_packed_cascade_layout_and_argument_errors():
    L = pkv.lib()
    offs = (ctypes.c_size_t * 11)()
    total = ctypes.c_size_t(0)
    B = 100
    assert L.pkv_packed_cascade_layout(B, 32, 8, 128, 256, pkv.BF16, pkv.BF16, offs,
                                       ctypes.byref(total)) == 0
    sizes = [B * 32 * 128 * 2, B * 8 * 128 * 2, B * 8 * 128 * 2, B * 256 * 4, B * 4,
             B * 4, B * 4, (B + 1) * 4, B * 4, B * 4,
             (B // 2) * 256 * 4]  # the step's inputs, then the groups and their page ids
    expect, o = [], 0
    for n in sizes:
        expect.append(o)
        o += (n + 255) // 256 * 256
    assert list(offs) == expect and total.value == o
    step = (ctypes.c_size_t * 5)()
    t5 = ctypes.c_size_t(0)
    L.pkv_packed_step_layout(B, 32, 8, 128, 256, pkv.BF16, pkv.BF16, step, ctypes.byref(t5))
    assert list(step) == expect[:5]  # the step's regions sit where the plain step has them
    d = _desc(cache_dtype=pkv.BF16)
    d.head_dim = 128
    fake = ctypes.c_void_p(1 << 20)
    assert L.pkv_cascade_decode_step_packed(None, fake, 2, 8, pkv.BF16, pkv.BF16, fake, fake,
                                            ctypes.byref(d), 4, 0.1, fake, fake, None, 0, None,
                                            None, None) == -1  # null host block


def test_empty_batches_need_no_buffers():
    # nothing to do: PKV_OK before any buffer (all NULL here) is looked at or anything launched
    L = pkv.lib()
    d = _desc(cache_dtype=pkv.BF16, head_dim=128)
    assert L.pkv_paged_decode_attention(None, pkv.BF16, 0, 4, None, None, ctypes.byref(d), None,
                                        16, None, 0.125, None, None, None, None, 0, None) == 0
    assert L.pkv_paged_decode_step(None, pkv.BF16, 0, 4, None, None, pkv.BF16, None, None,
                                   ctypes.byref(d), None, 16, None, 0.125, None, None, None,
                                   None, 0, None) == 0
    assert L.pkv_paged_decode_step_packed(None, None, 0, 4, pkv.BF16, pkv.BF16, None, None,
                                          ctypes.byref(d), 16, 0.125, None, None, 0, 0, None,
                                          None, None, 0, None) == 0
    n = ctypes.c_int32(-1)
    assert L.pkv_cascade_decode_step_packed(None, None, 0, 4, pkv.BF16, pkv.BF16, None, None,
                                            ctypes.byref(d), 16, 0.125, None, None, None, 0,
                                            None, ctypes.byref(n), None) == 0
    # a batch with work still needs its buffers
    assert L.pkv_paged_decode_step_packed(None, None, 1, 4, pkv.BF16, pkv.BF16, None, None,
                                          ctypes.byref(d), 16, 0.125, None, None, 0, 0, None,
                                          None, None, 0, None) == -1
