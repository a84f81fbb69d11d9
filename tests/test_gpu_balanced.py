"""The balanced split of the tensor-core decode against the oracle, and against the chunked split.

The balanced split cuts the whole call's (request, KV head, page) stream into equal shares, one
per warp of one wave of CTAs; a (request, KV head) that several warps share is merged from their
partials by the combine kernel. Cases cover: requests split over many warps and many requests in
one warp's share, requests with no pages, more warps than pages (empty shares), windows,
narrow caches with bf16 and fp32 queries, every group size, the fused append, and the error
word."""
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
    pkv.decode_set_split(2)
    pkv.device_error()
    yield
    pkv.decode_set_split(0)
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_merge_in_place(0)


def _err(out, ref):
    return float(np.abs(out.double().cpu().numpy() - ref).max()) if ref.size else 0.0


SHAPES = [
    # kv dtype, q dtype, h_q, h_kv, context lengths
    ("bf16", "bf16", 32, 8, [1, 16, 17, 31, 32, 33, 511, 512, 513, 1000]),
    ("bf16", "bf16", 64, 8, [300, 2049, 17]),
    ("bf16", "bf16", 8, 8, [700, 5, 1300, 64]),            # group 1
    ("bf16", "bf16", 32, 16, [250, 900]),                   # group 2
    ("bf16", "bf16", 16, 1, [1200, 3, 400]),                # group 16
    ("bf16", "bf16", 32, 8, [1] * 31 + [1500]),             # more warps than pages
    ("fp8_e4m3", "bf16", 32, 8, [40, 700, 1, 2000]),
    ("fp8_e4m3", "f32", 16, 1, [500, 19, 1111]),
    ("int8", "bf16", 32, 8, [40, 700, 1, 1100]),
    ("int8", "f32", 32, 4, [77, 260, 1600]),
]


@pytest.mark.parametrize("kv,qd,h_q,h_kv,lens", SHAPES)
def test_balanced_split_matches_oracle_and_chunks(kv, qd, h_q, h_kv, lens):
    w = workloads.custom("balanced", 15000 + h_q + 3 * h_kv + len(lens), len(lens), h_q, h_kv,
                         128, kv, qd, lens)
    sc = Scenario(w)
    sc.append()
    out = sc.decode().clone()
    again = sc.decode().clone()  # a second call on the same workspace
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out, again)
    ref = oracle_expected(w)
    err = _err(out, ref)
    assert err <= tolerance(w), err
    pkv.decode_set_split(1)
    chunked = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert _err(chunked, ref) <= tolerance(w)
    assert float((out.float() - chunked.float()).abs().max()) <= 2 * tolerance(w)


def test_balanced_split_leaves_the_workspace_for_an_in_place_merge():
    # the balanced split leaves the words the in-place merge counts chunks with untouched
    w = workloads.custom("balanced_then_inplace", 15101, 6, 32, 8, 128, "bf16", "bf16",
                         [900, 40, 1700, 3, 600, 1200])
    sc = Scenario(w)
    sc.append()
    sc.decode()
    pkv.decode_set_split(1)
    pkv.decode_set_merge_in_place(4096)
    out = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert _err(out, oracle_expected(w)) <= tolerance(w)


def test_balanced_split_with_empty_requests():
    w = workloads.custom("balanced_empty", 15102, 5, 32, 8, 128, "bf16", "bf16",
                         [600, 40, 900, 30, 2000])
    sc = Scenario(w)
    sc.append()
    cl = sc.context_lens.clone()
    cl[1] = 0
    cl[3] = 0
    out = pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables, cl, w.scale,
                                     workspace=sc.workspace)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert int(torch.count_nonzero(out[1])) == 0 and int(torch.count_nonzero(out[3])) == 0
    pairs = [(b, h) for b in (0, 2, 4) for h in range(32)]
    ref = oracle_expected(w, pairs=pairs)
    got = out.float().cpu().numpy()[[b for b, _ in pairs], [h for _, h in pairs]]
    assert float(np.abs(got - ref).max()) <= 1e-2


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_balanced_split_at_its_batch_limit(kv):
    # 2048 requests: the most page offsets the balanced split holds in shared memory
    rng = np.random.default_rng(15650)
    lens = [int(x) for x in rng.integers(1, 200, size=2048)]
    lens[100] = 1500
    lens[2047] = 1100
    w = workloads.custom("balanced_2048", 15650 + len(kv), len(lens), 32, 8, 128, kv, "bf16", lens)
    sc = Scenario(w)
    out = sc.fused_step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    pairs = ([(100, h) for h in range(32)] + [(2047, h) for h in range(32)] +
             [(b, (3 * b) % 32) for b in range(0, 2048, 37)])
    ref = oracle_expected(w, pairs=pairs)
    got = out.float().cpu().numpy()[[b for b, _ in pairs], [h for _, h in pairs]]
    assert float(np.abs(got - ref).max()) <= tolerance(w)


def test_balanced_split_above_its_batch_limit_takes_the_chunks():
    # the balanced split keeps the requests' page offsets in shared memory, for at most 2048
    # requests; a larger batch with the balanced split forced runs the chunks, bit for bit
    rng = np.random.default_rng(15600)
    lens = [int(x) for x in rng.integers(1, 48, size=2049)]
    lens[7] = 1100  # a table 69 pages wide: two chunk slots
    w = workloads.custom("balanced_big_batch", 15600, len(lens), 32, 8, 128, "bf16", "bf16", lens)
    sc = Scenario(w)
    sc.append()
    out = sc.decode().clone()
    pkv.decode_set_split(1)
    chunked = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out, chunked)
    pairs = [(7, h) for h in range(32)] + [(b, (5 * b) % 32) for b in range(0, 2049, 41)]
    ref = oracle_expected(w, pairs=pairs)
    got = out.float().cpu().numpy()[[b for b, _ in pairs], [h for _, h in pairs]]
    assert float(np.abs(got - ref).max()) <= tolerance(w)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "int8"])
def test_balanced_fused_step_equals_append_then_decode(kv):
    lens = [1, 2000, 33, 700, 16, 1500, 900, 64]
    w = workloads.custom("balanced_step", 15200 + len(kv), len(lens), 32, 8, 128, kv, "bf16", lens)
    a = Scenario(w)
    out_a = a.step().clone()
    b = Scenario(w)
    out_b = b.fused_step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert torch.equal(a.cache.v.view(torch.uint8), b.cache.v.view(torch.uint8))
    assert _err(out_b, oracle_expected(w)) <= tolerance(w)


@pytest.mark.parametrize("sink,window", [(4, 1024), (0, 100), (20, 40)])
def test_balanced_window(sink, window):
    lens = [3000, 1100, 50, 2500, 1024, 4000]
    w = workloads.custom("balanced_window", 15300 + window, len(lens), 32, 8, 128, "bf16", "bf16",
                         lens)
    sc = Scenario(w)
    out = sc.fused_step(window=window, sink_tokens=sink).clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    err = _err(out, oracle_expected(w, sink=sink, window=window))
    assert err <= 1e-2, err


def test_balanced_llama3_8b_batch64_full_parity():
    # every (request, query head) of the Llama-3-8B batch-64 layer under the balanced split
    w = workloads.llama3_8b_batch64()
    sc = Scenario(w)
    out = sc.step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    err = _err(out, oracle_expected(w))
    assert err <= 1e-2, err


def test_balanced_flags_bad_pages_and_cut_contexts():
    w = workloads.custom("balanced_bad", 15400, 3, 32, 8, 128, "bf16", "bf16", [400, 900, 60])
    sc = Scenario(w)
    sc.append()
    bt = sc.block_tables.clone()
    bt[1, 7] = w.num_pages + 3
    pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, bt, sc.context_lens, w.scale,
                               workspace=sc.workspace)
    assert pkv.device_error() & pkv.DEVERR_BAD_PAGE
    cl = sc.context_lens.clone()
    cl[2] = 16 * sc.block_tables.shape[1] + 40
    pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables, cl, w.scale,
                               workspace=sc.workspace)
    assert pkv.device_error() & pkv.DEVERR_BAD_PAGE
    # a clean call on the same workspace is right again
    out = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert _err(out, oracle_expected(w)) <= 1e-2


def test_autotuned_split_is_one_of_the_candidates_and_is_kept():
    pkv.decode_set_split(0)
    pkv.decode_autotune_reset()
    lens = [3000, 40, 1800, 700, 2500, 90, 1200, 4000]
    w = workloads.custom("balanced_tune", 15500, len(lens), 32, 8, 128, "fp8_e4m3", "bf16", lens)
    sc = Scenario(w)
    sc.append()
    maxp = sc.block_tables.shape[1]
    key = (torch.float8_e4m3fn, torch.bfloat16, w.batch, 32, 8, maxp)
    assert pkv.decode_split_choice(*key) == -1
    try:
        pkv.decode_set_autotune(True)
        tuned = sc.decode().clone()
        choice = pkv.decode_split_choice(*key)
        assert choice in (0, 1, 2, 3)
        again = sc.decode().clone()  # the recorded split, no timing
    finally:
        pkv.decode_set_autotune(False)
    pkv.decode_set_split({0: 1, 1: 2, 2: 3, 3: 4}[choice])  # the same split, forced
    fixed = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(tuned, again) and torch.equal(tuned, fixed)
    assert _err(tuned, oracle_expected(w)) <= tolerance(w)
    pkv.decode_autotune_reset()
    assert pkv.decode_split_choice(*key) == -1


def test_autotune_does_not_time_inside_graph_capture():
    # a shape first seen while its stream is captured: no timing (no synchronisation inside the
    # capture); the call takes chunks, and the graph replays to the chunked result
    pkv.decode_set_split(0)
    pkv.decode_autotune_reset()
    lens = [2200, 300, 1700, 60]
    w = workloads.custom("balanced_capture", 15501, len(lens), 32, 8, 128, "bf16", "bf16", lens)
    sc = Scenario(w)
    sc.append()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    try:
        pkv.decode_set_autotune(True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            sc.decode(stream=side)
        g.replay()
        torch.cuda.synchronize()
        captured = sc.out.clone()
        assert pkv.decode_split_choice(torch.bfloat16, torch.bfloat16, w.batch, 32, 8,
                                       sc.block_tables.shape[1]) == -1
    finally:
        pkv.decode_set_autotune(False)
    pkv.decode_set_split(1)
    chunked = sc.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(captured, chunked)


@pytest.mark.parametrize("mode", [3, 4], ids=["chunks_x1.5", "chunks_x2"])
@pytest.mark.parametrize("kv,qd,h_q,h_kv,lens", [
    ("bf16", "bf16", 32, 8, [1, 16, 17, 31, 32, 33, 511, 512, 513, 1000, 3000]),
    ("fp8_e4m3", "bf16", 32, 8, [40, 700, 1, 2000, 5000]),
    ("int8", "f32", 32, 4, [77, 260, 1600]),
    ("bf16", "bf16", 64, 8, [300, 2049, 17]),
])
def test_longer_chunks_match_oracle_and_fused_step(mode, kv, qd, h_q, h_kv, lens):
    # chunks 1.5 or 2 times the automatic length, in the same partial slots
    w = workloads.custom("longer_chunks", 15900 + h_q + len(lens), len(lens), h_q, h_kv, 128, kv,
                         qd, lens)
    pkv.decode_set_split(mode)
    a = Scenario(w)
    out_a = a.step().clone()
    b = Scenario(w)
    out_b = b.fused_step().clone()
    again = b.decode().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out_a, out_b) and torch.equal(out_b, again)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert _err(out_b, oracle_expected(w)) <= tolerance(w)


@pytest.mark.parametrize("mode", [3, 4])
def test_longer_chunks_window(mode):
    lens = [3000, 1100, 50, 2500, 1024, 4000]
    w = workloads.custom("longer_window", 15950 + mode, len(lens), 32, 8, 128, "bf16", "bf16",
                         lens)
    pkv.decode_set_split(mode)
    sc = Scenario(w)
    out = sc.fused_step(window=1024, sink_tokens=4).clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert _err(out, oracle_expected(w, sink=4, window=1024)) <= 1e-2
