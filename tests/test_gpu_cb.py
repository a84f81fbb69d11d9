"""FP8 E4M3 (and INT8) cache under continuous batching, against the oracle: per-head absmax scales,
quantising appends, requests finishing and being replaced (pages freed and reused through the
allocator), paged decode each step. Bit-exact scales and appended codes; attention within
1e-2 of the oracle's attention over its own dequantised codes."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import ContinuousBatchingRun

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


def _check_appended_codes(run, ks, vs):
    """The codes just written for each request's new token equal the oracle's quantiser."""
    t = run.t
    quant = oracle.quantize_int8 if run.cache_dtype == "int8" else oracle.quantize_e4m3
    slots = run.last_slots
    kc = run.cache.k.view(-1, t.num_kv_heads, 16, t.head_dim)
    for b in range(0, t.batch, max(1, t.batch // 8)):
        rid = run.slot_rid[b]
        p = run.cache.lens[rid] - 1
        s = int(slots[b])
        got = kc[s // 16, :, s % 16, :].cpu().numpy()
        x = run.tokens[rid][0][p].float().numpy()
        ref = np.stack([quant(x[j], ks[j]) for j in range(t.num_kv_heads)])
        np.testing.assert_array_equal(got, ref)


def _run(trace, pairs_per_step, full_check, cache_dtype="fp8_e4m3"):
    run = ContinuousBatchingRun(trace, cache_dtype=cache_dtype)
    k0, v0 = run.initial_rows()
    qmax = 127.0 if cache_dtype == "int8" else 448.0
    ks = oracle.absmax_scales_per_head(k0, qmax)
    vs = oracle.absmax_scales_per_head(v0, qmax)
    del k0, v0
    np.testing.assert_array_equal(run.k_scales.cpu().numpy(), ks)
    np.testing.assert_array_equal(run.v_scales.cpu().numpy(), vs)
    rng = np.random.default_rng(7)
    worst = 0.0
    freed_and_reused = 0
    for s in range(trace.steps):
        out = run.step()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        if full_check:
            pairs = [(b, h) for b in range(trace.batch) for h in range(trace.num_q_heads)]
        else:
            # every head of the longest live request, plus random (request, head) pairs
            lens = [run.cache.lens[r] for r in run.slot_rid]
            longest = int(np.argmax(lens))
            pairs = [(longest, h) for h in range(trace.num_q_heads)]
            pairs += [(int(rng.integers(trace.batch)), int(rng.integers(trace.num_q_heads)))
                      for _ in range(pairs_per_step)]
        ref = run.oracle_pairs(pairs, ks, vs)
        got = np.stack([out[b, h].double().cpu().numpy() for b, h in pairs])
        worst = max(worst, float(np.abs(got - ref).max()))
        _check_appended_codes(run, ks, vs)
        live = sum(len(run.cache.pages[r]) for r in run.slot_rid)
        assert run.cache.allocator.num_free() + live == trace.num_pages
        if s > 0:
            freed_and_reused += int(trace.finish[s - 1].sum())
    assert worst <= 1e-2, worst
    return freed_and_reused


def test_fp8_continuous_batching_small_full_check():
    tr = workloads.fp8_continuous_batching(batch=16, steps=8, lo=128, hi=512, rep_lo=16,
                                           rep_hi=400, p_finish=0.3)
    assert _run(tr, 0, full_check=True) > 0


def test_fp8_continuous_batching_full_size_sampled():
    tr = workloads.fp8_continuous_batching()
    assert _run(tr, 6, full_check=False) > 0


def test_int8_continuous_batching_small_full_check():
    tr = workloads.fp8_continuous_batching(batch=16, steps=8, lo=128, hi=512, rep_lo=16,
                                           rep_hi=400, p_finish=0.3)
    assert _run(tr, 0, full_check=True, cache_dtype="int8") > 0


def test_int8_continuous_batching_full_size_sampled():
    tr = workloads.fp8_continuous_batching(steps=6)
    assert _run(tr, 6, full_check=False, cache_dtype="int8") > 0


@pytest.mark.parametrize("split", [2, 3, 4], ids=["balanced", "chunks_x1.5", "chunks_x2"])
def test_fp8_continuous_batching_small_full_check_other_splits(split):
    pkv.decode_set_split(split)
    try:
        tr = workloads.fp8_continuous_batching(batch=16, steps=8, lo=128, hi=512, rep_lo=16,
                                               rep_hi=400, p_finish=0.3)
        assert _run(tr, 0, full_check=True) > 0
    finally:
        pkv.decode_set_split(0)


def test_fp8_continuous_batching_batch64_balanced_sampled():
    # the batch-64 trace, where the balanced split is the measured choice
    pkv.decode_set_split(2)
    try:
        tr = workloads.fp8_continuous_batching(batch=64, steps=5)
        assert _run(tr, 6, full_check=False) > 0
    finally:
        pkv.decode_set_split(0)
