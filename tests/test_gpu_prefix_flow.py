"""Prefix cache, request tables and cascade decode together ("KV cache and PagedAttention",
section 6: a prompt's pages are hashed, cached and reused by later requests with the same
prefix; here the reuse also shares the work of reading them). The first request writes a
prompt and registers its full pages; later requests of the same tenant start on those pages
(the lookup's references become theirs), write the prompt's partial last page and their own
tokens; the grouping finds the shared physical pages and the cascade decode must equal the
attention over each request's whole token sequence, computed by the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
from paged_kv_cache_271_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu

P, H_KV, G, D = 16, 4, 4, 128


def test_prefix_cache_requests_through_the_cascade_decode():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    g = torch.Generator().manual_seed(2710)
    rnd = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    prompt = list(range(5000, 5000 + 70))  # 4 full pages and 6 tokens
    pk, pv = rnd(len(prompt), H_KV, D), rnd(len(prompt), H_KV, D)
    n_req = 6
    own = [int(x) for x in torch.randint(1, 40, (n_req,), generator=g)]
    ok, ov = [rnd(n, H_KV, D) for n in own], [rnd(n, H_KV, D) for n in own]
    cache = PagedKVCache(256, H_KV, D, torch.bfloat16)
    pc = pkv.PrefixCache(cache.allocator, P)
    keys, vals = [], []
    for r in range(n_req):
        cached = cache.add_request_from_prefix_cache(r, pc, 3, prompt)
        assert cached == (0 if r == 0 else 64)
        rest_k = torch.cat([pk[cached:], ok[r]])  # the prompt past the cached pages, then own
        rest_v = torch.cat([pv[cached:], ov[r]])
        slots = cache.reserve([r], [rest_k.shape[0]])
        cache.write(slots, rest_k.cuda(), rest_v.cuda())
        if r == 0:
            cache.register_prompt(0, pc, 3, prompt)
        keys.append(torch.cat([pk, ok[r]]))
        vals.append(torch.cat([pv, ov[r]]))
    rids = list(range(n_req))
    assert all(cache.pages[r][:4] == cache.pages[0][:4] for r in rids)  # one copy of the prompt
    bt_h, cl_h = cache.block_table_array(rids), cache.context_lens_array(rids)
    groups = pkv.cascade_groups(bt_h, cl_h)
    assert groups.n_groups == 1 and list(groups.prefix_pages) == [4]
    q = rnd(n_req, H_KV * G, D)
    pkv.device_error()
    out = pkv.cascade_decode_attention(q.cuda(), cache.k, cache.v, torch.from_numpy(bt_h).cuda(),
                                       torch.from_numpy(cl_h).cuda(), D ** -0.5,
                                       groups.to("cuda"))
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    for r in rids:
        K, V, Q = keys[r].double().numpy(), vals[r].double().numpy(), q[r].double().numpy()
        ref = np.stack([oracle.attend(Q[h], K[:, h // G], V[:, h // G], D ** -0.5)
                        for h in range(H_KV * G)])
        assert float(np.abs(out[r].double().cpu().numpy() - ref).max()) < 1e-2, r
    cache.free_many(rids)
    assert pc.evict(4) == 4 and cache.allocator.num_free() == 256
