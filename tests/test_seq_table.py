"""Request page tables (pkv_seq_*) against a plain Python model, no GPU.

"KV cache and PagedAttention", sections 4-6 and 8; "KV Cache" glossary (shared blocks for
parallel sampling and beam search): a request is a row of pages plus a token count; forks share
pages by reference counts; a write into a shared, partly filled page copies it first; pages
wholly outside a sliding window go back to the pool. The model below does each operation the
obvious way on the oracle's allocator model, transactionally (a batch that runs out of pages is
undone by restoring a copy of the state), so the library's all-or-nothing pre-pass is checked
against plain replay rather than restated."""
import copy

import numpy as np
import pytest

import oracle
import paged_kv_cache_271_gb300 as pkv

P = 16


class SeqModel:
    def __init__(self, num_pages, order):
        self.a = oracle.AllocatorModel(num_pages, order)
        self.rows, self.lens = {}, {}

    def add(self, rid, shared=(), shared_len=0):
        if rid in self.rows or shared_len != len(shared) * P:
            raise ValueError
        self.a.incref(list(shared))
        self.rows[rid], self.lens[rid] = list(shared), shared_len

    def fork(self, srcs, news):
        for s, n in zip(srcs, news):
            if s not in self.rows or n in self.rows:
                raise ValueError
            self.rows[n] = list(self.rows[s])
            self.lens[n] = self.lens[s]
            self.a.incref([p for p in self.rows[n] if p >= 0])

    def free(self, rids):
        if len(set(rids)) != len(rids) or any(r not in self.rows for r in rids):
            raise ValueError
        for r in rids:
            self.a.decref([p for p in self.rows.pop(r) if p >= 0])
            del self.lens[r]

    def reserve(self, rids, counts):
        if len(set(rids)) != len(rids) or any(r not in self.rows for r in rids):
            raise ValueError
        slots, copies = [], []
        for r, n in zip(rids, counts):
            row = self.rows[r]
            if n > 0:
                lp = self.lens[r] // P
                if lp < len(row):
                    page = row[lp]
                    if page < 0:
                        raise ValueError
                    if self.a.ref[page] > 1:  # shared: a fresh page, one reference less here
                        fresh = self.a.alloc(1)[0]
                        self.a.ref[page] -= 1
                        row[lp] = fresh
                        copies.append((page, fresh))
            need = -(-(self.lens[r] + n) // P) - len(row)
            if need > 0:
                row += self.a.alloc(need)
            for k in range(n):
                pos = self.lens[r] + k
                slots.append(row[pos // P] * P + pos % P)
            self.lens[r] += n
        return slots, copies

    def release(self, rid, window, sink):
        n, row, gone = self.lens[rid], self.rows[rid], []
        if window > 0:
            for lp, pid in enumerate(row):
                if pid < 0:
                    continue
                positions = range(lp * P, min(lp * P + P, n))
                if all(t >= sink and t < n - window and t != n - 1 for t in positions):
                    gone.append(pid)
                    row[lp] = -1
        self.a.decref(gone)
        return len(gone)


def _same(model, table, alloc, num_pages):
    assert sorted(table.ids()) == sorted(model.rows)
    for r in model.rows:
        assert table.pages(r) == model.rows[r], r
        assert table.length(r) == model.lens[r], r
    assert [alloc.refcount(p) for p in range(num_pages)] == model.a.ref
    assert alloc.num_free() == model.a.num_free()


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_seq_table_against_model(seed):
    rng = np.random.default_rng(seed)
    num_pages = 48
    order = rng.permutation(num_pages)
    alloc = pkv.PageAllocator(num_pages, order)
    table = pkv.SeqTable(alloc, P)
    model = SeqModel(num_pages, order)
    next_id = 0
    ops = {"add": 0, "add_shared": 0, "fork": 0, "free": 0, "reserve": 0, "reserve_fail": 0,
           "copies": 0, "release": 0}
    for _ in range(600):
        live = sorted(model.rows)
        kind = rng.choice(["add", "fork", "free", "reserve", "reserve", "reserve", "release"])
        if kind == "add" or not live:
            rid = next_id
            next_id += 1
            donors = [r for r in live if model.lens[r] >= P and -1 not in model.rows[r]]
            if donors and rng.random() < 0.5:  # start on a prefix of another request's pages
                d = int(rng.choice(donors))
                k = int(rng.integers(1, model.lens[d] // P + 1))
                shared = model.rows[d][:k]
                model.add(rid, shared, k * P)
                table.add(rid, shared, k * P)
                ops["add_shared"] += 1
            else:
                model.add(rid)
                table.add(rid)
                ops["add"] += 1
        elif kind == "fork":
            m = int(rng.integers(1, 4))
            srcs, news = [], []
            for j in range(m):  # a parent may be forked earlier in the same call
                pool = live + news
                srcs.append(int(rng.choice(pool)))
                news.append(next_id)
                next_id += 1
            model.fork(srcs, news)
            table.fork(srcs, news)
            ops["fork"] += 1
        elif kind == "free":
            k = int(rng.integers(1, min(3, len(live)) + 1))
            rids = [int(x) for x in rng.choice(live, size=k, replace=False)]
            model.free(rids)
            table.free(rids)
            ops["free"] += 1
        elif kind == "reserve":
            k = int(rng.integers(1, min(6, len(live)) + 1))
            rids = [int(x) for x in rng.choice(live, size=k, replace=False)]
            counts = [int(rng.choice([0, 1, 1, 1, 3, 17, 40])) for _ in rids]
            saved = copy.deepcopy(model)
            try:
                want = model.reserve(rids, counts)
            except (MemoryError, ValueError):
                model = saved  # the batch does not fit (or writes into a released page)
                with pytest.raises(pkv.PkvError):
                    table.reserve(rids, counts)
                ops["reserve_fail"] += 1
            else:
                slots, copies = table.reserve(rids, counts)
                assert slots.tolist() == want[0]
                assert copies == want[1]
                ops["reserve"] += 1
                ops["copies"] += len(copies)
        else:
            rid = int(rng.choice(live))
            window, sink = int(rng.choice([0, 5, 20, 40])), int(rng.choice([0, 4, 16]))
            assert table.release_outside_window(rid, window, sink) == model.release(rid, window,
                                                                                     sink)
            ops["release"] += 1
        _same(model, table, alloc, num_pages)
    # the walk reached every branch
    assert all(v > 0 for v in ops.values()), ops
    table.free(sorted(model.rows))
    assert alloc.num_free() == num_pages


def test_seq_table_tables_and_errors():
    alloc = pkv.PageAllocator(8)
    t = pkv.SeqTable(alloc, P)
    t.add(5)
    t.add(7)
    s, c = t.reserve([5, 7], [20, 3])
    assert c == [] and len(s) == 23
    bt = t.tables([7, 5], 3)
    assert bt.tolist() == [t.pages(7) + [0, 0], t.pages(5) + [0]]
    assert t.lengths([5, 7]).tolist() == [20, 3]
    with pytest.raises(pkv.PkvError):
        t.tables([5], 1)  # two pages do not fit one column
    with pytest.raises(pkv.PkvError):
        t.reserve([5, 5], [1, 1])  # listed twice
    with pytest.raises(pkv.PkvError):
        t.reserve([9], [1])  # unknown
    with pytest.raises(pkv.PkvError):
        t.add(5)  # exists
    with pytest.raises(pkv.PkvError):
        t.add(6, t.pages(5), 20)  # not whole pages
    with pytest.raises(pkv.PkvError):
        t.fork([5], [7])  # exists
    with pytest.raises(pkv.PkvError):
        t.free([5, 5])
    free0 = alloc.num_free()
    with pytest.raises(pkv.PkvError):
        t.reserve([5, 7], [16, 16 * 8])  # more pages than the pool has: nothing changes
    assert alloc.num_free() == free0 and t.lengths([5, 7]).tolist() == [20, 3]
    # a released page cannot take a write: reserve refuses instead of writing through -1
    t.reserve([7], [13])  # 16 tokens: one full page
    t.fork([7], [8])
    assert t.release_outside_window(8, 1, 0) == 0  # the newest token's page stays
    t.free([5, 7, 8])
    assert alloc.num_free() == 8


def test_prefix_cache_and_request_tables_compose():
    # a prompt's full pages go into the prefix cache; a later request of the same tenant starts
    # on them (the lookup's references become the request's); freeing and evicting returns
    # every page to the pool
    import torch
    from paged_kv_cache_271_gb300.cache import PagedKVCache
    c = PagedKVCache(32, 2, 64, torch.float32, device="cpu")
    pc = pkv.PrefixCache(c.allocator, P)
    prompt = list(range(1000, 1050))  # 50 tokens: 3 full pages and 2 tokens
    assert c.add_request_from_prefix_cache(0, pc, 7, prompt) == 0  # nothing cached yet
    c.reserve([0], [len(prompt)])
    c.register_prompt(0, pc, 7, prompt)
    shared = c.pages[0][:3]
    assert [c.allocator.refcount(p) for p in shared] == [2, 2, 2]  # request 0 and the cache
    assert c.add_request_from_prefix_cache(1, pc, 7, prompt) == 48
    assert c.pages[1] == shared and c.lens[1] == 48
    assert [c.allocator.refcount(p) for p in shared] == [3, 3, 3]
    slots = c.reserve([1], [len(prompt) - 48 + 1])  # the rest of the prompt and one new token
    assert len(c.pages[1]) == 4 and c.pages[1][3] not in c.pages[0]
    assert all(s // P == c.pages[1][3] for s in slots)
    assert c.add_request_from_prefix_cache(2, pc, 8, prompt) == 0  # another tenant: no match
    c.free_many([0, 1, 2])
    assert [c.allocator.refcount(p) for p in shared] == [1, 1, 1]  # the cache's own
    assert pc.evict(3) == 3 and c.allocator.num_free() == 32
