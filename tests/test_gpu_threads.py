"""Decode calls from several host threads at once, each on its own stream.

The library's launch caches (shared-memory attributes, resident-CTA counts) and the split
autotuner's records are shared by all callers; these tests run calls of different shapes and
cache dtypes concurrently, with autotuning on, and check every result against the oracle and
against the same split forced afterwards on one thread (the kernels are deterministic, so the
two agree bit for bit)."""
import threading

import numpy as np
import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario, oracle_expected, tolerance

pytestmark = pytest.mark.gpu

FORCE = {0: 1, 1: 2, 2: 3, 3: 4}  # recorded split kind -> the split mode that forces it


@pytest.fixture(autouse=True)
def _modes():
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_merge_in_place(0)
    pkv.decode_set_split(0)
    pkv.decode_autotune_reset()
    pkv.device_error()
    yield
    pkv.decode_set_autotune(False)
    pkv.decode_set_split(0)
    pkv.decode_autotune_reset()


def _run_threads(fns):
    start = threading.Barrier(len(fns))
    errors = []

    def body(fn):
        try:
            start.wait(timeout=60)
            fn()
        except BaseException as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=body, args=(fn,)) for fn in fns]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a decode thread did not finish"
    if errors:
        raise errors[0]


def test_concurrent_decodes_with_autotuning():
    cases = [
        ("bf16", "bf16", [3000, 40, 1800, 700, 2500, 90, 1200, 4000]),
        ("fp8_e4m3", "bf16", [500, 2200, 17, 3100, 800, 60]),
        ("int8", "f32", [77, 2600, 1600, 900]),
        ("bf16", "bf16", [1, 16, 17, 2049, 513, 1000, 3333]),
    ]
    scs, streams, outs = [], [], []
    for i, (kv, qd, lens) in enumerate(cases):
        w = workloads.custom("threads", 16000 + i, len(lens), 32, 8, 128, kv, qd, lens)
        sc = Scenario(w)
        sc.append()
        scs.append(sc)
        streams.append(torch.cuda.Stream())
        outs.append(None)
    torch.cuda.synchronize()

    def worker(i):
        def fn():
            sc, s = scs[i], streams[i]
            with torch.cuda.stream(s):
                for _ in range(12):
                    sc.decode(stream=s)
                s.synchronize()
                outs[i] = sc.out.clone()
                s.synchronize()
        return fn

    pkv.decode_set_autotune(True)
    try:
        _run_threads([worker(i) for i in range(len(cases))])
    finally:
        pkv.decode_set_autotune(False)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    for i, sc in enumerate(scs):
        w = sc.w
        ref = oracle_expected(w)
        err = float(np.abs(outs[i].double().cpu().numpy() - ref).max())
        assert err <= tolerance(w), (i, err)
        choice = pkv.decode_split_choice(sc.cache.k.dtype, sc.q.dtype, w.batch, 32, 8,
                                         sc.block_tables.shape[1])
        if choice < 0:  # a shape with a single split: nothing was timed
            pkv.decode_set_split(1)
        else:
            pkv.decode_set_split(FORCE[choice])
        again = sc.decode().clone()
        torch.cuda.synchronize()
        pkv.decode_set_split(0)
        assert torch.equal(outs[i], again), i


def test_concurrent_fused_steps_on_one_shape():
    # four threads, the same shape (so the same launch cache entries and one autotune record),
    # separate caches: every thread's pool bytes and outputs equal a single-threaded run
    lens = [1200, 33, 2600, 700, 1, 1900]
    ws = [workloads.custom("threads_same", 16100 + i, len(lens), 32, 8, 128, "fp8_e4m3", "bf16",
                           lens) for i in range(4)]
    scs = [Scenario(w) for w in ws]
    streams = [torch.cuda.Stream() for _ in ws]
    outs = [None] * len(ws)
    torch.cuda.synchronize()

    def worker(i):
        def fn():
            s = streams[i]
            with torch.cuda.stream(s):
                outs[i] = scs[i].fused_step(stream=s).clone()
                s.synchronize()
        return fn

    pkv.decode_set_autotune(True)
    try:
        _run_threads([worker(i) for i in range(len(ws))])
    finally:
        pkv.decode_set_autotune(False)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    choice = pkv.decode_split_choice(torch.float8_e4m3fn, torch.bfloat16, len(lens), 32, 8,
                                     scs[0].block_tables.shape[1], fused=True)
    pkv.decode_set_split(FORCE[choice] if choice >= 0 else 1)
    for i, w in enumerate(ws):
        ref_sc = Scenario(w)
        ref_out = ref_sc.fused_step().clone()
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref_out), i
        assert torch.equal(scs[i].cache.k.view(torch.uint8), ref_sc.cache.k.view(torch.uint8))
        assert torch.equal(scs[i].cache.v.view(torch.uint8), ref_sc.cache.v.view(torch.uint8))
        err = float(np.abs(outs[i].double().cpu().numpy() - oracle_expected(w)).max())
        assert err <= tolerance(w), (i, err)
