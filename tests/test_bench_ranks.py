"""The benchmark's multi-rank logic on CPU: two gloo ranks, replicas with a max-over-ranks
step time and a whole-job aggregate. No GPU and no data-path collective."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    ws, r, _ = bench.rank_info()
    local_ms = 1.0 + r  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    bench.barrier()
    q.put((r, ws, m, bench.aggregate(1e9, m, ws)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, ws, m, agg in res:
        assert ws == 2 and m == 2.0
        # 2 ranks x 1 GB each over the slowest rank's 2 ms = 1000 GB/s
        assert agg == pytest.approx(1000.0)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate(2e9, 2.0, 1) == pytest.approx(1000.0)


def test_bench_cli_and_workload_configs_without_gpu():
    import workloads
    for name in ("llama3_8b_b64", "llama3_70b_long", "prefix_sharing"):
        if name == "llama3_70b_long":
            continue  # large draw; same code path as the others
        cfg = bench.config_of(bench.workload(name))
        assert cfg["workload"] and cfg["kv_dtype"] == "bf16"
    assert set(bench.WORKLOADS) >= {"llama3_8b_b64", "fp8_cb_b256"}
    w = workloads.llama3_8b_batch64()
    # the metric's bytes: the sum of the drawn context lengths times 8 heads x 128 dims x 2 B x 2
    assert bench.config_of(w)["context_lens"].endswith(str(int(w.context_lens.sum())))


def test_trace_joins_follow_the_request_table():
    import workloads
    tr = workloads.fp8_continuous_batching(batch=32, steps=12, lo=128, hi=512, p_finish=0.2)
    joins = bench.trace_joins(tr)
    assert joins[0] == [] and sum(len(j) for j in joins) == int(tr.finish[:-1].sum()) > 0
    seen = set(range(tr.batch))
    for s in range(1, tr.steps):
        live = list(tr.rid_table[s - 1])
        for b, old, new in joins[s]:
            assert tr.finish[s - 1, b] and old == live[b] and new not in seen
            live[b] = new
            seen.add(new)
        assert live == list(tr.rid_table[s])  # every other slot keeps its request
    assert sorted(seen) == list(range(len(tr.prompt_lens)))  # ids 0, 1, ... in join order


def test_trace_bookkeeping_full_size_matches_the_trace():
    # the bench's per-step bookkeeping over the whole 256-slot trace, host only: incrementally
    # patched tables equal a full export, lengths equal each request's position + 1, and the
    # prompts get exactly their token counts of distinct slots
    import torch
    import paged_kv_cache_271_gb300 as pkv
    from paged_kv_cache_271_gb300.cache import PagedKVCache
    import workloads
    tr = workloads.fp8_continuous_batching(steps=35)
    B = tr.batch
    cache = PagedKVCache(tr.num_pages, 1, 16, torch.uint8, device="cpu",
                         initial_free_order=tr.page_order)
    for b in range(B):
        cache.add_request(b)
    cache.reserve(list(range(B)), [int(x) for x in tr.initial_lens])
    joins = bench.trace_joins(tr)
    width = pkv.pages_needed(int(tr.prompt_lens.max()) + tr.steps)
    bt = torch.zeros((B, width), dtype=torch.int32)
    cl = torch.zeros(B, dtype=torch.int32)
    rid_arr = np.arange(B, dtype=np.int64)
    start = {b: 0 for b in range(B)}
    for s in range(tr.steps):
        for _, _, r in joins[s]:
            start[r] = s
        slots = bench.trace_bookkeeping(cache, tr, joins[s], rid_arr, width, bt, cl)
        assert rid_arr.tolist() == [int(r) for r in tr.rid_table[s]]
        want = [int(tr.prompt_lens[r]) + s - start[r] + 1 for r in tr.rid_table[s]]
        assert cl.tolist() == want
        assert np.array_equal(bt.numpy(), cache.block_table_array(rid_arr, width))
        n = sum(int(tr.prompt_lens[r]) for _, _, r in joins[s])
        assert len(slots) == n and len(set(slots.tolist())) == n
    assert cache.allocator.num_free() + sum(len(cache.pages[r]) for r in rid_arr.tolist()) \
        == tr.num_pages
