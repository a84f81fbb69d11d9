"""A fused decode step captured once in a CUDA graph and replayed over several decode steps.

Serving loops replay one captured step per layer; between replays only the contents of the
captured buffers change: this step's queries and K/V rows, the page tables (a request that
crosses a page boundary gets a new page) and the lengths (one more token each step). Every
split must read those contents at replay time -- the balanced split's stream offsets are
worked out inside the decode from the lengths, the chunked grids cover the table width -- so
each replay must equal the same step run eagerly, bit for bit, in outputs and pool bytes."""
import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _modes():
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_merge_in_place(0)
    pkv.decode_set_split(0)
    pkv.decode_set_autotune(False)
    pkv.device_error()
    yield
    pkv.decode_set_split(0)


def _widen(sc, width):
    sc.block_tables = torch.from_numpy(sc.cache.block_table_array(sc.rids, width)).to(sc.device)
    w = sc.w
    need = pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, width)
    sc.workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=sc.device)


@pytest.mark.parametrize("split", [1, 2, 3, 4], ids=["chunks", "balanced", "chunks_x1.5",
                                                     "chunks_x2"])
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("sink,window", [(0, 0), (4, 256)], ids=["full", "window"])
def test_graph_replayed_steps_follow_the_tables_and_lengths(kv, split, sink, window):
    lens = [15, 16, 31, 700, 1000, 2047, 2048, 33]
    w = workloads.custom("graph_steps", 16500 + split + 10 * len(kv) + window, len(lens), 32, 8,
                         128, kv, "bf16", lens)
    pkv.decode_set_split(split)
    a, b = Scenario(w), Scenario(w)
    width = a.block_tables.shape[1] + 2  # room for the pages the steps below add
    _widen(a, width)
    _widen(b, width)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        b.fused_step(stream=side, window=window, sink_tokens=sink)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(16500 + split)
    B, h_kv, d = w.batch, w.num_kv_heads, w.head_dim
    for step in range(20):
        if step > 0:
            q = torch.randn(b.q.shape, generator=gen, device="cuda").to(b.q.dtype)
            kr = torch.randn((B, h_kv, d), generator=gen, device="cuda").to(b.k_new.dtype)
            vr = torch.randn((B, h_kv, d), generator=gen, device="cuda").to(b.v_new.dtype)
            for sc in (a, b):
                sc.cache.reserve(sc.rids, [1] * B)
            bt = torch.from_numpy(b.cache.block_table_array(b.rids, width)).to(b.device)
            cl = torch.from_numpy(b.cache.context_lens_array(b.rids)).to(b.device)
            a.q, a.k_new, a.v_new = q.clone(), kr.clone(), vr.clone()
            a.block_tables = torch.from_numpy(a.cache.block_table_array(a.rids, width)).to(a.device)
            a.context_lens = torch.from_numpy(a.cache.context_lens_array(a.rids)).to(a.device)
            b.q.copy_(q)
            b.k_new.copy_(kr)
            b.v_new.copy_(vr)
            b.block_tables.copy_(bt)
            b.context_lens.copy_(cl)
            torch.cuda.synchronize()
        eager = a.fused_step(window=window, sink_tokens=sink).clone()
        g.replay()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.equal(eager, b.out), step
        assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8)), step
        assert torch.equal(a.cache.v.view(torch.uint8), b.cache.v.view(torch.uint8)), step
