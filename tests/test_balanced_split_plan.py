"""The balanced split's plan, restated on the host and checked for the properties its kernels
rely on (the GPU tests check the kernels themselves against the oracle).

The plan: the call's pages form one stream -- every (request b, KV head j, attended page p) in
order b, j, p; with T pages and N warps, warp w takes stream pages [w T / N, (w + 1) T / N);
each run of one (b, j)'s pages in a share is a segment, which writes the output when it is the
whole of (b, j) and otherwise the partial numbered w + r (r = b h_kv + j); a share that is
empty but falls inside a (b, j) (not at its first page) leaves an empty partial there; the
combine merges, for each (b, j), the partials owner(P0) + r .. owner(P0 + n - 1) + r in order,
owner(P) being the last w with w T / N <= P. Checked here: every page is attended exactly once
and in stream order within its (b, j); the partial numbers are distinct and below N + B h_kv;
the combine's run for each (b, j) is exactly the set of partials written for it; the page-id
lookup of a warp's k-th page agrees with its segment walk."""
import random

import pytest

PAGE = 16


def walked_pages(ctx, sink, window):
    pages = (ctx + PAGE - 1) // PAGE
    if window > 0:
        first_window_page = max(0, ctx - window) // PAGE
        sink_pages = min((max(0, sink) + PAGE - 1) // PAGE, pages)
        if first_window_page > sink_pages:
            return sink_pages + (pages - first_window_page)
    return pages


def request_of(pre, F, h_kv):
    """The last b with pre[b] * h_kv <= F."""
    q = F // h_kv
    lo, hi = 0, len(pre) - 2
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if pre[mid] <= q:
            lo = mid
        else:
            hi = mid - 1
    return lo


def owner(P, T, N):
    return ((P + 1) * N + T - 1) // T - 1


def locate(pre, F, h_kv):
    b = request_of(pre, F, h_kv)
    nb = pre[b + 1] - pre[b]
    off = F - pre[b] * h_kv
    return b, off // nb, off % nb


def plan(ctxs, h_kv, N, sink=0, window=0):
    """What the decode writes: outputs {r: pages}, partials {id: (r, pages)}."""
    B = len(ctxs)
    pre = [0]
    for c in ctxs:
        pre.append(pre[-1] + walked_pages(c, sink, window))
    T = pre[B] * h_kv
    outputs, partials = {}, {}
    for w in range(N):
        s0, s1 = w * T // N, (w + 1) * T // N
        if s0 >= s1:
            if s0 < T:
                b, j, p = locate(pre, s0, h_kv)
                if p > 0:
                    assert w + b * h_kv + j not in partials
                    partials[w + b * h_kv + j] = (b * h_kv + j, [])
            continue
        b, j, p = locate(pre, s0, h_kv)
        nb = pre[b + 1] - pre[b]
        m, n_mine = 0, s1 - s0
        while m < n_mine:
            p_end = min(nb, p + (n_mine - m))
            r = b * h_kv + j
            pages = []
            for pp in range(p, p_end):
                assert locate(pre, s0 + m, h_kv) == (b, j, pp)  # the page-id lookup
                pages.append(s0 + m)
                m += 1
            if p == 0 and p_end == nb:
                assert r not in outputs
                outputs[r] = pages
            else:
                assert w + r not in partials
                partials[w + r] = (r, pages)
            p = p_end
            if p == nb:
                p, j = 0, j + 1
                if j == h_kv:
                    j, b = 0, b + 1
                    while b < B - 1 and pre[b + 1] == pre[b]:
                        b += 1
                nb = pre[b + 1] - pre[b] if b < B else 0
    return pre, T, outputs, partials


def check(ctxs, h_kv, N, sink=0, window=0):
    pre, T, outputs, partials = plan(ctxs, h_kv, N, sink, window)
    B, R = len(ctxs), len(ctxs) * h_kv
    covered, read = [], set()
    for r in range(R):
        b, j = divmod(r, h_kv)
        nb = pre[b + 1] - pre[b]
        row = list(range(pre[b] * h_kv + j * nb, pre[b] * h_kv + (j + 1) * nb))
        if nb == 0:
            assert r not in outputs
            continue
        first = owner(row[0], T, N)
        count = owner(row[-1], T, N) - first + 1
        if count == 1:
            assert outputs.get(r) == row
            covered += row
            continue
        assert r not in outputs
        got = []
        for k in range(count):
            pid = first + r + k
            assert pid in partials and partials[pid][0] == r
            read.add(pid)
            got += partials[pid][1]
        assert got == row  # stream order
        covered += got
    assert covered == list(range(T))
    assert read == set(partials)
    assert all(pid < N + R for pid in partials)


@pytest.mark.parametrize("seed", range(6))
def test_balanced_split_plan_random_layouts(seed):
    rng = random.Random(seed)
    for _ in range(60):
        B = rng.choice([1, 2, 3, 8, 33, 64])
        h_kv = rng.choice([1, 2, 8])
        N = rng.choice([4, 12, 100, 1824])
        kind = rng.random()
        if kind < 0.2:
            ctxs = [rng.choice([0, 0, 1, 16, 17]) for _ in range(B)]
        elif kind < 0.6:
            ctxs = [rng.randint(0, 300) for _ in range(B)]
        else:
            ctxs = [rng.randint(0, 8192) for _ in range(B)]
        if not any(ctxs):
            ctxs[0] = 5
        window = rng.choice([0, 0, 64, 1024])
        sink = rng.choice([0, 4, 20]) if window else 0
        check(ctxs, h_kv, N, sink, window)


def test_balanced_split_plan_edge_layouts():
    check([0, 0, 0, 7], 8, 1824)            # more warps than pages: empty shares
    check([1] * 63 + [4000], 1, 1824)       # one long request among single pages
    check([4096] * 4, 8, 4)                 # every share inside one (b, j)
    check([16] * 128, 8, 1024)              # shares that start exactly on (b, j) boundaries
