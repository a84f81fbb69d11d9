"""Copy-on-write fork (pages shared across sequences for parallel sampling or beam search,
"KV Cache" glossary): forked requests share their parent's pages; the first write into a
shared, partly filled page copies it. Each request must still attend exactly its own history."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
from paged_kv_cache_271_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    pkv.device_error()


@pytest.mark.parametrize("prompt", [40, 48, 1])
def test_forked_requests_diverge_correctly(prompt):
    g = torch.Generator().manual_seed(11 + prompt)
    h_kv, d, h_q, n_children, steps = 4, 128, 16, 3, 20
    rows = lambda n: torch.randn(n, h_kv, d, generator=g).to(torch.bfloat16)
    cache = PagedKVCache(64, h_kv, d, torch.bfloat16, "cuda")
    cache.k.fill_(float("nan"))
    cache.v.fill_(float("nan"))
    cache.add_request(0)
    pk, pv = rows(prompt), rows(prompt)
    cache.write(cache.reserve([0], [prompt]), pk.cuda(), pv.cuda())
    hist = {0: (pk, pv)}
    for c in range(1, n_children + 1):
        cache.fork(0, c)
        hist[c] = (pk, pv)
    shared_full = prompt // 16
    for p in cache.pages[0][:shared_full]:
        assert cache.allocator.refcount(p) == n_children + 1
    rids = list(range(n_children + 1))
    for _ in range(steps):  # every sequence appends its own tokens
        kn, vn = rows(len(rids)), rows(len(rids))
        slots = cache.reserve(rids, [1] * len(rids))
        cache.write(slots, kn.cuda(), vn.cuda())
        for i, r in enumerate(rids):
            hist[r] = (torch.cat([hist[r][0], kn[i:i + 1]]), torch.cat([hist[r][1], vn[i:i + 1]]))
    assert pkv.device_error() == 0
    # the full prompt pages are still shared; every other page belongs to one request
    for p in cache.pages[0][:shared_full]:
        assert cache.allocator.refcount(p) == n_children + 1
    owners = {}
    for r in rids:
        for p in cache.pages[r][shared_full:]:
            owners.setdefault(p, []).append(r)
    assert all(len(v) == 1 for v in owners.values())
    q = torch.randn(len(rids), h_q, d, generator=g).to(torch.bfloat16)
    bt = torch.from_numpy(cache.block_table_array(rids)).cuda()
    cl = torch.from_numpy(cache.context_lens_array(rids)).cuda()
    out = pkv.paged_decode_attention(q.cuda(), cache.k, cache.v, bt, cl, d ** -0.5)
    assert pkv.device_error() == 0
    K = torch.cat([hist[r][0] for r in rids])
    V = torch.cat([hist[r][1] for r in rids])
    lens = np.array([hist[r][0].shape[0] for r in rids], dtype=np.int32)
    off = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    ref = oracle.contiguous_decode(oracle.as_raw(q, "bf16"), "bf16", oracle.as_raw(K, "bf16"),
                                   oracle.as_raw(V, "bf16"), "bf16", off, lens, d ** -0.5)
    assert float(np.abs(out.double().cpu().numpy() - ref).max()) <= 1e-2
    for r in rids:
        cache.free_request(r)
    assert cache.allocator.num_free() == 64
