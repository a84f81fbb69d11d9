"""The allocation-free decode entry point (pkv_paged_decode_attention_noalloc), called through
the C ABI, against the regular entry point that takes a caller workspace.

It exists for callers that cannot allocate device memory (a plugin inside an application that
owns all device memory, a server whose KV pools took all free HBM, a loop that must not risk
cudaMalloc's device-wide synchronisation). This file is collected last on purpose."""
import ctypes

import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    pkv.decode_set_chunk_pages(0)
    pkv.device_error()
    yield
    pkv.decode_set_chunk_pages(0)


def _noalloc(sc, q, out):
    desc = pkv.cache_desc(sc.cache.k)
    st = pkv.lib().pkv_paged_decode_attention_noalloc(
        ctypes.c_void_p(q.data_ptr()), pkv.BF16, q.shape[0], q.shape[1],
        ctypes.c_void_p(sc.cache.k.data_ptr()), ctypes.c_void_p(sc.cache.v.data_ptr()),
        ctypes.byref(desc), ctypes.c_void_p(sc.block_tables.data_ptr()),
        sc.block_tables.shape[1], ctypes.c_void_p(sc.context_lens.data_ptr()),
        ctypes.c_float(sc.w.scale), None, None, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pkv.lib().pkv_last_error().decode()


@pytest.mark.parametrize("merge", ["combine kernel", "merge in place", "balanced split"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(merge):
    # split partials merged by the combine kernel, or by the last CTA of each (request, KV
    # head) through the chunk counters, or the balanced split's partials in their own region:
    # every use of the scratch
    import dataclasses
    from gpu_harness import oracle_expected
    w = workloads.llama3_8b_batch64(batch=8)
    sc = Scenario(w)
    sc.append()
    need = pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     sc.block_tables.shape[1])
    assert 0 < need <= pkv.lib().pkv_decode_noalloc_scratch_bytes()  # the split scratch is used
    q2 = (sc.q.float() * -0.7).to(torch.bfloat16)
    if merge == "balanced split":
        pkv.decode_set_split(2)
    else:
        pkv.decode_set_chunk_pages(8)  # several chunks per request
    pkv.decode_set_merge_in_place(64 if merge == "merge in place" else 0)
    try:
        need = pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                         sc.block_tables.shape[1])
        assert need <= pkv.lib().pkv_decode_noalloc_scratch_bytes()
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        for q in (sc.q, q2):  # the second call must not see the first call's leftovers
            ref = pkv.paged_decode_attention(q, sc.cache.k, sc.cache.v, sc.block_tables,
                                             sc.context_lens, w.scale, workspace=ws).clone()
            out = torch.full_like(q, float("nan"))
            _noalloc(sc, q, out)
            torch.cuda.synchronize()
            assert pkv.device_error() == 0
            assert torch.equal(out, ref)  # same kernels, same split: the same bits
            exp = oracle_expected(dataclasses.replace(w, q=q.cpu()))
            err = float((out.double().cpu() - torch.from_numpy(exp)).abs().max())
            assert err <= 1e-2, err
    finally:
        pkv.decode_set_chunk_pages(0)
        pkv.decode_set_merge_in_place(0)
        pkv.decode_set_split(0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fake = ctypes.c_void_p(1 << 20)  # never touched: the size check fails before any launch
    desc = pkv._Desc(70000, 16, 8, 128, pkv.BF16)
    st = pkv.lib().pkv_paged_decode_attention_noalloc(fake, pkv.BF16, 64, 32, fake, fake,
                                                      ctypes.byref(desc), fake, 4096, fake,
                                                      ctypes.c_float(0.088), None, None, fake,
                                                      None)
    assert st == -1
    assert "scratch" in pkv.lib().pkv_last_error().decode()
