"""The README's usage example, run as written (small sizes), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
from paged_kv_cache_271_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu


def test_readme_example():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    g = torch.Generator().manual_seed(271)
    prompt_len, scale = 700, 128 ** -0.5
    k_prompt = torch.randn(prompt_len, 8, 128, generator=g).to(torch.bfloat16)
    v_prompt = torch.randn(prompt_len, 8, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 32, 128, generator=g).to(torch.bfloat16)
    k_new = torch.randn(1, 8, 128, generator=g).to(torch.bfloat16)
    v_new = torch.randn(1, 8, 128, generator=g).to(torch.bfloat16)

    cache = PagedKVCache(num_pages=4096, num_kv_heads=8, head_dim=128, dtype=torch.bfloat16)
    cache.add_request(0)
    slots = cache.reserve([0], [prompt_len])
    cache.write(slots, k_prompt.cuda(), v_prompt.cuda())
    cache.reserve([0], [1])
    bt = torch.from_numpy(cache.block_table_array([0])).cuda()
    cl = torch.from_numpy(cache.context_lens_array([0])).cuda()
    out = pkv.paged_decode_step(q.cuda(), k_new.cuda(), v_new.cuda(), cache.k, cache.v, bt, cl,
                                scale)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert int(cl[0]) == prompt_len + 1

    K = torch.cat([k_prompt, k_new]).double().numpy()  # [T, 8, 128]
    V = torch.cat([v_prompt, v_new]).double().numpy()
    Q = q.double().numpy()[0]
    ref = np.stack([oracle.attend(Q[h], K[:, h // 4], V[:, h // 4], scale) for h in range(32)])
    assert float(np.abs(out[0].double().cpu().numpy() - ref).max()) <= 1e-2
