"""Sliding-window decode with attention sinks ("KV cache and PagedAttention", section 8) against
the oracle: only the last W positions plus the first S are attended; pages holding none of them
are never read, so they can be released."""
import numpy as np
import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario, oracle_expected, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True)
def _defaults():
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_split(0)
    pkv.device_error()
    yield
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_split(0)


CASES = [
    ("bf16", "bf16", 32, 8, 128, [1, 17, 300, 1200, 2049]),
    ("f32", "f32", 4, 2, 64, [18, 34, 100]),
    ("fp8_e4m3", "bf16", 32, 8, 128, [40, 700, 1, 1000]),
    ("int8", "bf16", 32, 8, 128, [40, 700, 1, 1000]),
]
WINDOWS = [(0, 1), (0, 16), (4, 64), (16, 100), (3, 500), (0, 4096)]


@pytest.mark.parametrize("kv,qd,h_q,h_kv,d,lens", CASES)
@pytest.mark.parametrize("sink,window", WINDOWS)
@pytest.mark.parametrize("kernel,chunk,split", [(1, 0, 0), (2, 0, 0), (2, 3, 0), (2, 0, 2)],
                         ids=["cuda_cores", "tensor_cores", "tensor_cores_chunk3", "balanced"])
def test_window_decode_parity(kv, qd, h_q, h_kv, d, lens, sink, window, kernel, chunk, split):
    if kernel == 2 and (kv == "f32" or d != 128):
        pytest.skip("the tensor-core decode serves bf16/FP8 caches with head_dim 128")
    w = workloads.custom("win", 5000 + h_q + len(lens), len(lens), h_q, h_kv, d, kv, qd, lens)
    pkv.decode_set_kernel(kernel)
    pkv.decode_set_chunk_pages(chunk)
    pkv.decode_set_split(split)
    sc = Scenario(w)
    out = sc.fused_step(window=window, sink_tokens=sink).clone()
    assert pkv.device_error() == 0
    ref = oracle_expected(w, sink=sink, window=window)
    err = float(np.abs(out.double().cpu().numpy() - ref).max())
    assert err <= tolerance(w), err


# (split: 1 chunks, 2 balanced, 3 and 4 chunks 1.5 and 2 times longer)
@pytest.mark.parametrize("kernel,split", [(1, 1), (2, 1), (2, 2), (2, 3), (2, 4)])
def test_released_pages_are_never_read(kernel, split):
    w = workloads.custom("winrel", 5101, 6, 32, 8, 128, "bf16", "bf16",
                         [40, 700, 1000, 2049, 1, 513])
    pkv.decode_set_kernel(kernel)
    pkv.decode_set_split(split)
    sink, window = 4, 100
    sc = Scenario(w)
    full = sc.fused_step(window=window, sink_tokens=sink).clone()
    before = {r: list(sc.cache.pages[r]) for r in sc.rids}
    released = sum(sc.cache.release_outside_window(r, window, sink) for r in sc.rids)
    assert released > 0
    sc.refresh_tables()
    assert int((sc.block_tables < 0).sum()) == released
    gone = [p for r in sc.rids for p, q in zip(before[r], sc.cache.pages[r]) if q < 0]
    idx = torch.tensor(gone, device="cuda")
    sc.cache.k[idx] = float("nan")  # stale contents of pages handed back to the allocator
    sc.cache.v[idx] = float("nan")
    # released pages get junk (and may be handed out again): results must not change
    again = sc.fused_step(window=window, sink_tokens=sink).clone()
    assert pkv.device_error() == 0
    assert torch.equal(full, again)
    ref = oracle_expected(w, sink=sink, window=window)
    assert float(np.abs(again.double().cpu().numpy() - ref).max()) <= 1e-2


def test_window_argument_errors():
    w = workloads.custom("winerr", 5102, 2, 8, 2, 64, "bf16", "bf16", [20, 9])
    sc = Scenario(w)
    with pytest.raises(pkv.PkvError):
        sc.fused_step(window=-1)
    with pytest.raises(pkv.PkvError):
        sc.fused_step(window=0, sink_tokens=4)


def test_windowed_host_step_equals_device_step():
    # the packed host-memory step with a window: one copy in, the windowed fused step, one out
    w = workloads.custom("hostwin", 7400, 4, 8, 2, 128, "bf16", "bf16", [300, 45, 1000, 17])
    a = Scenario(w)
    out_a = a.fused_step(window=64, sink_tokens=4).clone()
    b = Scenario(w)
    hs = pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                      b.block_tables.shape[1])
    hs.q_host.copy_(b.q.cpu())
    hs.k_new_host.copy_(b.k_new.cpu())
    hs.v_new_host.copy_(b.v_new.cpu())
    hs.block_tables_host.copy_(b.block_tables.cpu())
    hs.context_lens_host.copy_(b.context_lens.cpu())
    out_b = hs.step(b.cache.k, b.cache.v, w.scale, workspace=b.workspace, window=64,
                    sink_tokens=4)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out_a.cpu(), out_b)
    err = float(np.abs(out_b.double().numpy() - oracle_expected(w, sink=4, window=64)).max())
    assert err <= tolerance(w), err
