"""Failure detection in the kernels' waits: every copy and MMA barrier wait is bounded, gives
up after its limit and reports PKV_DEVERR_TIMEOUT instead of hanging. Here one wait runs out
on purpose (a barrier nothing completes), and the GPU context is shown to be usable after it."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    pkv.device_error()
    t0 = time.perf_counter()
    bits, done = pkv.selftest_wait_timeout()
    elapsed = time.perf_counter() - t0
    assert done == 1  # the wait gave up (2 would mean it completed)
    assert bits & pkv.DEVERR_TIMEOUT
    assert 1.5 < elapsed < 60, elapsed  # the limit is 2 s
    # the context still works: a library kernel afterwards, checked against the oracle
    g = torch.Generator().manual_seed(5)
    x = torch.randn(300, 2, 64, generator=g).to(torch.bfloat16)
    got = pkv.kv_absmax_scales(x.cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.absmax_scales_per_head(x.float().numpy(), 448.0))
    assert pkv.device_error() == 0  # the library's own word was not touched
