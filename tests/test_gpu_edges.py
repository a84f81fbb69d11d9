"""Buffers that start off a 16-byte boundary.

The tensor-core decode reads the query with 16-byte loads, so a query that starts elsewhere
takes the CUDA-core kernel (element loads); outputs are written element by element on every
path, at any element boundary. Pools, new rows and workspaces must be 16-byte aligned and are
refused on the host otherwise, before anything is launched."""
import numpy as np
import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario, oracle_expected, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _modes():
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_merge_in_place(0)
    pkv.decode_set_split(0)
    pkv.device_error()
    yield
    pkv.decode_set_split(0)
    pkv.decode_set_kernel(0)


def _err(out, ref):
    return float(np.abs(out.double().cpu().numpy() - ref).max())


def _offset_view(like, elems, fill=0):
    """A contiguous tensor shaped like `like` that starts `elems` elements into a larger buffer,
    and that buffer."""
    n = like.numel()
    buf = torch.full((n + 16,), fill, dtype=like.dtype, device=like.device)
    return buf[elems:elems + n].view(like.shape), buf


@pytest.mark.parametrize("split", [1, 2], ids=["chunks", "balanced"])
@pytest.mark.parametrize("kv,qd", [("bf16", "bf16"), ("fp8_e4m3", "bf16"), ("int8", "f32")])
@pytest.mark.parametrize("q_off,out_off", [(1, 3), (0, 1), (2, 0)])
def test_query_and_output_off_the_16_byte_boundary(kv, qd, q_off, out_off, split):
    lens = [1, 300, 2100, 17, 900, 3000]
    w = workloads.custom("unaligned", 16200 + q_off + 7 * out_off + len(kv), len(lens), 32, 8,
                         128, kv, qd, lens)
    pkv.decode_set_split(split)
    sc = Scenario(w)
    sc.append()
    q, _ = _offset_view(sc.q, q_off)
    q.copy_(sc.q)
    out, obuf = _offset_view(sc.q, out_off)
    ks, vs = sc.scales if sc.scales else (None, None)
    pkv.paged_decode_attention(q, sc.cache.k, sc.cache.v, sc.block_tables, sc.context_lens,
                               w.scale, out=out, k_scales=ks, v_scales=vs,
                               workspace=sc.workspace)
    aligned = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    ref = oracle_expected(w)
    assert _err(out, ref) <= tolerance(w)
    assert _err(aligned, ref) <= tolerance(w)
    if q_off % (16 // q.element_size()) == 0:  # the same kernel either way
        assert torch.equal(out, aligned)
    n = out.numel()  # nothing written outside the output
    assert int(torch.count_nonzero(obuf[:out_off])) == 0
    assert int(torch.count_nonzero(obuf[out_off + n:])) == 0


def test_fused_step_with_output_off_the_boundary_equals_the_aligned_one():
    lens = [700, 1, 2500, 64, 1300]
    w = workloads.custom("unaligned_step", 16300, len(lens), 32, 8, 128, "fp8_e4m3", "bf16", lens)
    a = Scenario(w)
    ref_out = a.fused_step().clone()
    b = Scenario(w)
    out, obuf = _offset_view(b.q, 5)
    ks, vs = b.scales
    pkv.paged_decode_step(b.q, b.k_new, b.v_new, b.cache.k, b.cache.v, b.block_tables,
                          b.context_lens, w.scale, out=out, k_scales=ks, v_scales=vs,
                          workspace=b.workspace)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert int(torch.count_nonzero(obuf[:5])) == 0
    assert int(torch.count_nonzero(obuf[5 + out.numel():])) == 0


def test_misaligned_rows_pools_and_workspace_are_refused_before_any_launch():
    lens = [400, 2000, 33]
    w = workloads.custom("unaligned_refused", 16400, len(lens), 32, 8, 128, "bf16", "bf16", lens)
    sc = Scenario(w)
    sc.append()
    before_k = sc.cache.k.view(torch.uint8).clone()
    k_new, _ = _offset_view(sc.k_new, 1)
    k_new.copy_(sc.k_new)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_step(sc.q, k_new, sc.v_new, sc.cache.k, sc.cache.v, sc.block_tables,
                              sc.context_lens, w.scale, workspace=sc.workspace)
    assert e.value.code == -4
    ws = torch.zeros(sc.workspace.numel() + 32, dtype=torch.uint8, device=sc.workspace.device)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables,
                                   sc.context_lens, w.scale, workspace=ws[8:8 + sc.workspace.numel()])
    assert e.value.code == -4
    pool = torch.zeros(sc.cache.k.numel() + 16, dtype=sc.cache.k.dtype, device=sc.cache.k.device)
    k_pool = pool[1:1 + sc.cache.k.numel()].view(sc.cache.k.shape)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(sc.q, k_pool, sc.cache.v, sc.block_tables, sc.context_lens,
                                   w.scale, workspace=sc.workspace)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(sc.cache.k.view(torch.uint8), before_k)  # the refused step wrote nothing


@pytest.mark.parametrize("split", [1, 2, 3, 4])
@pytest.mark.parametrize("kernel", [1, 2], ids=["cuda_cores", "tensor_cores"])
def test_every_context_empty(kernel, split):
    # a table wide enough to split, but no request has a token: zero outputs, nothing appended
    lens = [1200, 30, 2100, 5]
    w = workloads.custom("all_empty", 16600 + split, len(lens), 32, 8, 128, "bf16", "bf16", lens)
    pkv.decode_set_kernel(kernel)
    pkv.decode_set_split(split)
    sc = Scenario(w)
    zero = torch.zeros_like(sc.context_lens)
    k_before = sc.cache.k.view(torch.uint8).clone()
    out = torch.full_like(sc.q, 7.0)
    pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables, zero, w.scale,
                               out=out, workspace=sc.workspace)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert int(torch.count_nonzero(out)) == 0
    out.fill_(7.0)
    pkv.paged_decode_step(sc.q, sc.k_new, sc.v_new, sc.cache.k, sc.cache.v, sc.block_tables,
                          zero, w.scale, out=out, workspace=sc.workspace)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert int(torch.count_nonzero(out)) == 0
    assert torch.equal(sc.cache.k.view(torch.uint8), k_before)


def test_empty_batch_launches_nothing():
    w = workloads.custom("empty_batch", 16700, 2, 32, 8, 128, "bf16", "bf16", [300, 40])
    sc = Scenario(w)
    q = sc.q[:0]
    out = pkv.paged_decode_attention(q, sc.cache.k, sc.cache.v, sc.block_tables[:0],
                                     sc.context_lens[:0], w.scale)
    assert out.shape == q.shape
    out = pkv.paged_decode_step(q, sc.k_new[:0], sc.v_new[:0], sc.cache.k, sc.cache.v,
                                sc.block_tables[:0], sc.context_lens[:0], w.scale)
    torch.cuda.synchronize()
    assert out.shape == q.shape and pkv.device_error() == 0


@pytest.mark.parametrize("kernel,split", [(1, 1), (2, 1), (2, 2), (2, 3), (2, 4)])
def test_contexts_around_8192_tokens(kernel, split):
    # a partial last page (8191), exactly full pages (8192), one token onto a new page (8193)
    lens = [8191, 8192, 8193, 1, 15]
    w = workloads.custom("ctx8k", 16800 + 10 * kernel + split, len(lens), 32, 8, 128, "bf16",
                         "bf16", lens)
    pkv.decode_set_kernel(kernel)
    pkv.decode_set_split(split)
    sc = Scenario(w)
    out = sc.fused_step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert _err(out, oracle_expected(w)) <= tolerance(w)
