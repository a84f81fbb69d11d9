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


def _model_step(model, free, new, prompts, live):
    """pkv_seq_step on the model: frees stand; if the pages run out, the new requests are
    removed again (their pages returned in the library's order). Returns (prompt slots,
    copies) or None when the pages ran out."""
    model.free(free)
    for r in new:
        model.add(r)
    before = copy.deepcopy(model)
    out = None
    try:
        ps, c1 = model.reserve(new, prompts)
    except MemoryError:
        model.__dict__.update(before.__dict__)
    else:
        assert c1 == []
        mid = copy.deepcopy(model)
        try:
            out = ps, model.reserve(live, [1] * len(live))[1]
        except MemoryError:
            model.__dict__.update(mid.__dict__)
    if out is None:  # back to the state after the frees
        for r in new:
            model.a.decref([p for p in model.rows.pop(r) if p >= 0])
            del model.lens[r]
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_seq_step_against_model(seed):
    rng = np.random.default_rng(100 + seed)
    num_pages = 40
    order = rng.permutation(num_pages)
    alloc = pkv.PageAllocator(num_pages, order)
    table = pkv.SeqTable(alloc, P)
    model = SeqModel(num_pages, order)
    next_id, seen = 0, {"ok": 0, "nopages": 0, "copies": 0, "reuse": 0}
    for _ in range(300):
        live = sorted(model.rows)
        if live and rng.random() < 0.2:  # a fork between steps: shared pages, later copies
            src = int(rng.choice(live))
            model.fork([src], [next_id])
            table.fork([src], [next_id])
            next_id += 1
            _same(model, table, alloc, num_pages)
            continue
        k = int(rng.integers(0, min(3, len(live)) + 1))
        free = [int(x) for x in rng.choice(live, size=k, replace=False)] if k else []
        new = []
        if free and rng.random() < 0.2:  # a freed id comes back as a new request
            new.append(free[0])
            seen["reuse"] += 1
        for _ in range(int(rng.integers(0, 3))):
            new.append(next_id)
            next_id += 1
        prompts = [int(rng.choice([0, 1, 5, 16, 17, 40, 200, 400])) for _ in new]
        rest = [r for r in live if r not in free]
        keep = [r for r in rest if rng.random() < 0.85]
        live_now = keep + [r for r in new if rng.random() < 0.9]
        rng.shuffle(live_now)
        live_now = [int(r) for r in live_now]
        # a write into a released page is refused up front: keep such requests out
        live_now = [r for r in live_now if r in new or model.lens[r] // P >= len(model.rows[r])
                    or model.rows[r][model.lens[r] // P] >= 0]
        width = num_pages if rng.random() < 0.5 else None  # None: the library sizes the rows
        want = _model_step(model, free, new, prompts, live_now)
        if want is None:
            with pytest.raises(pkv.PkvError):
                table.step(free, new, prompts, live_now, width)
            seen["nopages"] += 1
        else:
            ps, bt, cl, copies = table.step(free, new, prompts, live_now, width)
            if width is None:  # the widest live row after the step, at least one column
                width = max([len(model.rows[r]) for r in live_now] + [1])
                assert bt.shape == (len(live_now), width)
            assert ps.tolist() == want[0] and copies == want[1]
            assert cl.tolist() == [model.lens[r] for r in live_now]
            for i, r in enumerate(live_now):
                row = model.rows[r]
                assert bt[i].tolist() == row + [0] * (width - len(row))
            seen["ok"] += 1
            seen["copies"] += len(copies)
        _same(model, table, alloc, num_pages)
    assert all(v > 0 for v in seen.values()), seen
    table.free(sorted(model.rows))
    assert alloc.num_free() == num_pages


def test_seq_step_checks_before_changing_anything():
    alloc = pkv.PageAllocator(8)
    t = pkv.SeqTable(alloc, P)
    t.add(1)
    t.add(2)
    t.reserve([1, 2], [20, 3])
    state = ([t.pages(r) for r in (1, 2)], t.lengths([1, 2]).tolist(), alloc.num_free())

    def same():
        assert ([t.pages(r) for r in (1, 2)], t.lengths([1, 2]).tolist(),
                alloc.num_free()) == state and sorted(t.ids()) == [1, 2]

    bad = [([9], [], [], [2]),            # unknown request to free
           ([1, 1], [], [], [2]),         # freed twice
           ([], [2], [4], [2]),           # a new id that is live
           ([], [5, 5], [1, 1], [5]),     # a new id listed twice
           ([1], [], [], [1]),            # a freed request decoded
           ([], [], [], [2, 2]),          # decoded twice
           ([], [], [], [7])]             # unknown live request
    for free, new, prompts, live in bad:
        with pytest.raises(pkv.PkvError):
            t.step(free, new, prompts, live, 8)
        same()
    with pytest.raises(pkv.PkvError):
        t.step([2], [], [], [1], 1)  # request 1 needs 2 columns: refused before the free
    same()
    # a freed id may come back as a new request in the same step
    ps, bt, cl, cp = t.step([2], [2], [5], [1, 2], 4)
    assert len(ps) == 5 and cl.tolist() == [21, 6] and cp == []
    # out of pages: the frees stand, the new requests are gone again
    free_before = alloc.num_free()
    with pytest.raises(pkv.PkvError):
        t.step([2], [3], [16 * 8], [1, 3], 16)
    assert sorted(t.ids()) == [1] and alloc.num_free() == free_before + 1
    t.free([1])
    assert alloc.num_free() == 8


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_seq_step_incremental_tables_stay_exact(seed):
    # one buffer across steps, rows patched in place: after every step it must equal the
    # model's rows; slots keep their requests (a replacement takes a finished one's row),
    # with shuffles, window releases, forks and a plain export into the same buffer mixed in
    rng = np.random.default_rng(200 + seed)
    num_pages = 48
    order = rng.permutation(num_pages)
    alloc = pkv.PageAllocator(num_pages, order)
    table = pkv.SeqTable(alloc, P)
    model = SeqModel(num_pages, order)
    width = num_pages
    buf = np.full((64, width), -7, dtype=np.int32)
    lens = np.zeros(64, dtype=np.int32)
    slots = []  # live request per row, in row order
    next_id = 0
    seen = {"patched": 0, "shuffle": 0, "release": 0, "plain": 0, "fork": 0, "nopages": 0}
    for _ in range(250):
        r = rng.random()
        if slots and r < 0.1:
            rid = int(rng.choice(slots))
            window, sink = int(rng.choice([5, 20, 40])), int(rng.choice([0, 4]))
            assert table.release_outside_window(rid, window, sink) == model.release(rid, window,
                                                                                     sink)
            seen["release"] += 1
        elif slots and r < 0.15:
            src = int(rng.choice(slots))
            model.fork([src], [next_id])
            table.fork([src], [next_id])
            slots.append(next_id)
            next_id += 1
            seen["fork"] += 1
        elif slots and r < 0.2:
            table.tables(slots, width, out=buf[:len(slots)])  # forgets the incremental state
            seen["plain"] += 1
        elif slots and r < 0.3:
            rng.shuffle(slots)
            seen["shuffle"] += 1
        k = int(rng.integers(0, min(2, len(slots)) + 1))
        free = [int(x) for x in rng.choice(slots, size=k, replace=False)] if k else []
        new = [next_id + i for i in range(int(rng.integers(0, 3)))]
        next_id += len(new)
        prompts = [int(rng.choice([0, 3, 16, 17, 40, 120, 400])) for _ in new]
        live = list(slots)
        for i, f in enumerate(free):  # a new request takes a finished one's row
            j = live.index(f)
            if i < len(new):
                live[j] = new[i]
            else:
                live[j] = None
        live = [x for x in live if x is not None] + new[len(free):]
        live = [x for x in live if x in new or model.lens[x] // P >= len(model.rows[x])
                or model.rows[x][model.lens[x] // P] >= 0]
        want = _model_step(model, free, new, prompts, live)
        if want is None:
            with pytest.raises(pkv.PkvError):
                table.step(free, new, prompts, live, width, buf[:len(live)], lens[:len(live)],
                           incremental=True)
            slots = [x for x in slots if x not in free]
            seen["nopages"] += 1
            _same(model, table, alloc, num_pages)
            continue
        ps, _, _, copies = table.step(free, new, prompts, live, width, buf[:len(live)],
                                      lens[:len(live)], incremental=True)
        assert ps.tolist() == want[0] and copies == want[1]
        slots = live
        for i, x in enumerate(slots):
            row = model.rows[x]
            assert buf[i].tolist() == row + [0] * (width - len(row)), (i, x)
            assert lens[i] == model.lens[x]
        seen["patched"] += 1
        _same(model, table, alloc, num_pages)
    assert all(v > 0 for v in seen.values()), seen


def test_seq_step_checks_its_host_buffers():
    alloc = pkv.PageAllocator(16)
    t = pkv.SeqTable(alloc, P)
    t.step([], [1, 2], [20, 3], [1, 2], width=4)
    for bad in (np.zeros((2, 3), np.int32), np.zeros((2, 4), np.int64),
                np.zeros((4, 2), np.int32).T, np.zeros((3, 4), np.int32)):
        with pytest.raises(pkv.PkvError):
            t.step([], [], [], [1, 2], width=4, tables_out=bad)
    with pytest.raises(pkv.PkvError):
        t.step([], [], [], [1, 2], width=4, lens_out=np.zeros(3, np.int32))
    assert t.lengths([1, 2]).tolist() == [21, 4]  # the refused calls changed nothing
    # incremental without a buffer of the caller's: every row is written in full
    for _ in range(3):
        _, bt, cl, _ = t.step([], [], [], [1, 2], width=4, incremental=True)
        assert bt.tolist() == [t.pages(1) + [0] * (4 - len(t.pages(1))),
                               t.pages(2) + [0] * (4 - len(t.pages(2)))]
    import torch
    out = torch.zeros(2, 4, dtype=torch.int32)
    _, bt, _, _ = t.step([], [], [], [1, 2], width=4, tables_out=out)
    assert bt is out and out[0].tolist()[:2] == t.pages(1)


def test_seq_step_judges_sharing_after_the_frees():
    # a forked child writes into the partly filled page it shares with its parent; when the
    # parent finishes in the same step, the page is the child's alone and needs no copy
    import ctypes
    alloc = pkv.PageAllocator(8)
    t = pkv.SeqTable(alloc, P)
    t.add(1)
    t.reserve([1], [20])  # one full page and a partly filled one
    L = pkv.lib()

    def step(free, live):
        f = np.array(free, np.int64)
        lv = np.array(live, np.int64)
        bt = np.zeros((len(live), 4), np.int32)
        cl = np.zeros(len(live), np.int32)
        nc = ctypes.c_int32(-1)
        st = L.pkv_seq_step(t._h, f.ctypes.data if f.size else None, f.size, None, None, 0,
                            None, lv.ctypes.data, lv.size, None, 4, bt.ctypes.data,
                            cl.ctypes.data, 0, None, None, ctypes.byref(nc))
        return st, nc.value

    t.fork([1], [2])
    before = (t.pages(2), alloc.num_free())
    st, _ = step([], [2])  # the parent lives on: the page is shared and there are no copy arrays
    assert st != 0 and (t.pages(2), alloc.num_free()) == before
    st, nc = step([1], [2])
    assert st == 0 and nc == 0 and t.pages(2) == before[0] and t.length(2) == 21
    assert [alloc.refcount(p) for p in t.pages(2)] == [1, 1]


def test_seq_step_width_query():
    alloc = pkv.PageAllocator(64)
    t = pkv.SeqTable(alloc, P)
    t.add(1)
    t.reserve([1], [31])  # 2 pages; one more token still fits
    t.add(2)
    t.reserve([2], [32])  # 2 full pages; one more token needs a third
    L = pkv.lib()

    def width(new, prompts, live):
        import ctypes
        n = np.array(new, np.int64)
        c = np.array(prompts, np.int32)
        lv = np.array(live, np.int64)
        w = ctypes.c_int32(0)
        st = L.pkv_seq_step_width(t._h, n.ctypes.data if n.size else None,
                                  c.ctypes.data if c.size else None, n.size,
                                  lv.ctypes.data if lv.size else None, lv.size, ctypes.byref(w))
        return w.value if st == 0 else None

    assert width([], [], []) == 1
    assert width([], [], [1]) == 2
    assert width([], [], [1, 2]) == 3
    assert width([5], [47], [1, 5]) == 3  # 48 tokens after the step: 3 pages
    assert width([5], [48], [5]) == 4     # 49 tokens: 4 pages
    assert width([], [], [9]) is None     # unknown request
