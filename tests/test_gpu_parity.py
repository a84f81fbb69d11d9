"""CUDA library vs the fp64 CPU oracle, through the C ABI, on seeded synthetic inputs.

Bit-exact for the append (bf16/fp32 copies and FP8 codes), slot mapping and FP8 scales;
attention output within 1e-5 max-abs for fp32 inputs and 1e-2 for bf16/FP8 inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import Scenario, fill_junk, oracle_expected, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_cache_271_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    yield
    pkv.decode_set_chunk_pages(0)


@pytest.fixture(autouse=True)
def _clean_error_word():
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_merge_in_place(0)
    pkv.device_error()
    yield
    pkv.decode_set_chunk_pages(0)
    pkv.decode_set_kernel(0)
    pkv.decode_set_merge_in_place(0)


def _max_err(out, ref):
    return float(np.abs(out.double().cpu().numpy() - ref).max()) if ref.size else 0.0


def _run(w, chunk=0, kernel=0, **kw):
    pkv.decode_set_chunk_pages(chunk)
    pkv.decode_set_kernel(kernel)
    sc = Scenario(w, **kw)
    out = sc.step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    return sc, out


# ---- the workloads ------------------------------------------------------------------------------

def test_tiny_ref_parity():
    w = workloads.tiny_ref()
    sc, out = _run(w)
    assert list(sc.context_lens.cpu().numpy()) == [18, 34]
    assert _max_err(out, oracle_expected(w)) <= 1e-5


def test_llama3_8b_batch64_parity_full():
    w = workloads.llama3_8b_batch64()
    sc, out = _run(w)
    err = _max_err(out, oracle_expected(w))
    assert err <= 1e-2, err


def test_llama3_70b_long_context_parity_full():
    # every (request, query head) pair: 4 x 64 outputs over contexts of up to 131072 tokens
    w = workloads.llama3_70b_long()
    sc, out = _run(w)
    err = _max_err(out, oracle_expected(w))
    assert err <= 1e-2, err
    # every output is a convex combination of value rows
    vmax = float(w.v_tokens.float().abs().max())
    assert bool(torch.isfinite(out).all()) and float(out.float().abs().max()) <= vmax


def test_prefix_sharing_parity_and_shared_equals_copied():
    w = workloads.prefix_sharing()
    sc, shared = _run(w, share_prefix=True)
    assert [sc.cache.allocator.refcount(p) for p in sc.shared_pages] == [w.batch] * 125
    err = _max_err(shared, oracle_expected(w))
    assert err <= 1e-2, err
    del sc
    torch.cuda.empty_cache()
    _, copied = _run(w, share_prefix=False)
    assert torch.equal(shared, copied)


# ---- shapes, dtypes, split-K and ragged tails ---------------------------------------------------

SHAPES = [
    # kv dtype, q dtype, h_q, h_kv, d, context lengths
    ("f32", "f32", 4, 2, 64, [18, 34]),
    ("f32", "f32", 8, 8, 128, [1, 15, 16, 17, 100]),
    ("f32", "f32", 16, 1, 64, [33, 200, 7]),
    ("bf16", "bf16", 32, 8, 128, [1, 16, 17, 31, 32, 33, 511, 512, 513, 1000]),
    ("bf16", "bf16", 64, 8, 128, [300, 2049, 17]),
    ("bf16", "bf16", 16, 16, 64, [45, 800]),
    ("bf16", "bf16", 32, 2, 64, [129, 3]),
    ("fp8_e4m3", "bf16", 32, 8, 128, [40, 700, 1]),
    ("fp8_e4m3", "f32", 8, 4, 64, [77, 260]),
    ("fp8_e4m3", "bf16", 16, 1, 128, [500, 19]),
    ("int8", "bf16", 32, 8, 128, [40, 700, 1, 1100]),
    ("int8", "f32", 16, 2, 64, [77, 260]),
]


@pytest.mark.parametrize("kv,qd,h_q,h_kv,d,lens", SHAPES)
@pytest.mark.parametrize("chunk", [0, 1, 3])
@pytest.mark.parametrize("kernel", [1, 2])  # CUDA-core, tensor-core
def test_decode_parity_shapes(kv, qd, h_q, h_kv, d, lens, chunk, kernel):
    pkv.decode_set_merge_in_place(16 if chunk == 3 else 0)
    if kernel == 2 and (kv == "f32" or d != 128):
        pytest.skip("the tensor-core decode serves bf16/FP8 caches with head_dim 128")
    w = workloads.custom("shape", 9000 + h_q + d + len(lens), len(lens), h_q, h_kv, d, kv, qd,
                         lens)
    _, out = _run(w, chunk=chunk, kernel=kernel)
    err = _max_err(out, oracle_expected(w))
    assert err <= tolerance(w), err


# FP8 and INT8 caches contract the query with widened codes in f16 on the tensor cores; f16
# holds neither bf16's nor fp32's range. Scaling q by 2^f and the softmax scale by 2^-f leaves
# the exact result unchanged, so every case below must match the oracle like the plain one.
@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("qd", ["bf16", "f32"])
@pytest.mark.parametrize("f", [16, -20, 100, -100])
@pytest.mark.parametrize("h_q,h_kv", [(32, 8), (16, 1)])
@pytest.mark.parametrize("kernel", [1, 2])
def test_narrow_cache_decode_for_any_query_range(kv, qd, f, h_q, h_kv, kernel):
    import dataclasses
    lens = [40, 700, 1, 300]
    w = workloads.custom("q_range", 9100 + h_q, len(lens), h_q, h_kv, 128, kv, qd, lens)
    qs = (w.q.double() * 2.0 ** f).to(w.q.dtype)
    assert torch.equal(qs.double() * 2.0 ** -f, w.q.double())  # the scaling is exact
    w = dataclasses.replace(w, q=qs, scale=w.scale * 2.0 ** -f)
    _, out = _run(w, chunk=1 if h_kv == 1 else 0, kernel=kernel)
    assert bool(torch.isfinite(out).all())
    err = _max_err(out, oracle_expected(w))
    assert err <= tolerance(w), err


def test_narrow_cache_fp32_query_keeps_its_precision():
    # an fp32 query is contracted as two f16 parts (22 significant bits): against a bf16
    # rounding of the same query, the fp32 one must land closer to the oracle of the fp32 query
    lens = [500, 1300, 64, 2000]
    w = workloads.custom("q_f32", 9200, len(lens), 32, 8, 128, "fp8_e4m3", "f32", lens)
    _, out = _run(w, kernel=2)
    err32 = _max_err(out, oracle_expected(w))
    import dataclasses
    wb = dataclasses.replace(w, q=w.q.to(torch.bfloat16).float())
    _, outb = _run(wb, kernel=2)
    errb = _max_err(outb, oracle_expected(w))
    assert err32 <= 1e-2 and err32 < errb, (err32, errb)


@pytest.mark.parametrize("chunk", [1, 2, 3])
@pytest.mark.parametrize("kernel", [1, 2])
def test_combine_of_many_chunks(chunk, kernel):
    # more than 16 chunk slots: each (request, head) is merged by four warps, each over a run
    # of consecutive chunks; requests with 1, 2, 3, 5, 17 and 63+ chunks leave some warps an
    # empty run
    lens = [1000, 16, 17, 33, 70, 260, 1, 2, 1500]
    w = workloads.custom("many_chunks", 9500 + chunk, len(lens), 16, 4, 128, "bf16", "bf16", lens)
    sc, out = _run(w, chunk=chunk, kernel=kernel)
    assert _max_err(out, oracle_expected(w)) <= tolerance(w)


@pytest.mark.parametrize("kernel", [1, 2])
def test_split_results_do_not_depend_on_physical_pages(kernel):
    w = workloads.llama3_8b_batch64(batch=8)
    _, a = _run(w, kernel=kernel)
    order2 = np.random.default_rng(5).permutation(w.num_pages).astype(np.int32)
    _, b = _run(w, kernel=kernel, page_order=order2)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", [1, 2])
def test_llama3_8b_batch64_both_kernels(kernel):
    w = workloads.llama3_8b_batch64(batch=16)
    _, out = _run(w, kernel=kernel)
    err = _max_err(out, oracle_expected(w))
    assert err <= 1e-2, err


STEP_SHAPES = [
    ("bf16", "bf16", 32, 8, 128, [1, 16, 17, 500, 1100, 2049]),
    ("int8", "bf16", 32, 8, 128, [3, 600, 16]),
    ("f32", "f32", 4, 2, 64, [18, 34, 1]),
    ("fp8_e4m3", "bf16", 32, 8, 128, [40, 700, 1, 1000]),
    ("fp8_e4m3", "f32", 16, 8, 128, [33, 129]),
]


@pytest.mark.parametrize("kv,qd,h_q,h_kv,d,lens", STEP_SHAPES)
@pytest.mark.parametrize("chunk,merge", [(0, 0), (0, 16), (5, 16), (1, 0)])
@pytest.mark.parametrize("kernel", [1, 2])
def test_fused_step_equals_append_then_decode(kv, qd, h_q, h_kv, d, lens, chunk, merge, kernel):
    if kernel == 2 and (kv == "f32" or d != 128):
        pytest.skip("the tensor-core decode serves bf16/FP8 caches with head_dim 128")
    w = workloads.custom("step", 7000 + h_q + len(lens), len(lens), h_q, h_kv, d, kv, qd, lens)
    pkv.decode_set_chunk_pages(chunk)
    pkv.decode_set_kernel(kernel)
    pkv.decode_set_merge_in_place(merge)
    a = Scenario(w)
    out_a = a.step().clone()
    b = Scenario(w)
    out_b = b.fused_step().clone()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert torch.equal(a.cache.v.view(torch.uint8), b.cache.v.view(torch.uint8))
    err = _max_err(out_b, oracle_expected(w))
    assert err <= tolerance(w), err
    # the workspace is left ready for the next call: a second step gives the same output
    out_c = b.fused_step().clone()
    assert torch.equal(out_b, out_c)


def test_tensor_core_kernel_rejects_what_it_cannot_serve():
    w = workloads.custom("f32mma", 41, 2, 4, 2, 64, "f32", "f32", [20, 9])
    sc = Scenario(w)
    pkv.decode_set_kernel(2)
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables,
                                   sc.context_lens, w.scale, workspace=sc.workspace)


def test_zero_length_context_gives_zero_output():
    w = workloads.custom("zero", 77, 3, 8, 2, 64, "bf16", "bf16", [5, 40, 3])
    sc = Scenario(w)
    sc.append()
    cl = sc.context_lens.clone()
    cl[1] = 0
    out = pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables, cl, w.scale,
                                     workspace=sc.workspace)
    assert pkv.device_error() == 0
    assert int(torch.count_nonzero(out[1])) == 0
    ref = oracle_expected(w, pairs=[(0, h) for h in range(8)])
    assert _max_err(out[0], ref) <= 1e-2


# ---- append, scales -------------------------------------------------------------------------------

@pytest.mark.parametrize("kv,src", [("f32", "f32"), ("bf16", "bf16"), ("fp8_e4m3", "bf16"),
                                     ("fp8_e4m3", "f32"), ("int8", "bf16"), ("int8", "f32")])
def test_append_bit_exact(kv, src):
    torch.manual_seed(0)
    num_pages, h_kv, d, N = 24, 4, 128, 150
    pool_dt = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
               "int8": torch.int8}[kv]
    src_dt = {"f32": torch.float32, "bf16": torch.bfloat16}[src]
    kc = torch.empty(num_pages, h_kv, 16, d, dtype=pool_dt, device="cuda")
    vc = torch.empty_like(kc)
    fill_junk(kc, 1)
    fill_junk(vc, 2)
    rng = np.random.default_rng(1)
    slots = rng.permutation(num_pages * 16)[:N].astype(np.int64)
    slots[::17] = -1  # padding rows are skipped
    kn = (torch.randn(N, h_kv, d) * 3).to(src_dt)
    vn = (torch.randn(N, h_kv, d) * 0.01).to(src_dt)
    raw = (lambda t: t.view(torch.uint8).cpu().numpy().copy())
    exp_k, exp_v = raw(kc), raw(vc)
    ks = vs = None
    if kv in ("fp8_e4m3", "int8"):
        quant = oracle.quantize_int8 if kv == "int8" else oracle.quantize_e4m3
        ks = torch.tensor([0.01, 0.02, 0.003, 1.0], device="cuda")
        vs = torch.tensor([1e-4, 2e-5, 3e-5, 0.5], device="cuda")
        kq = np.stack([quant(kn.float().numpy()[:, j], ks[j].item()) for j in range(h_kv)], 1)
        vq = np.stack([quant(vn.float().numpy()[:, j], vs[j].item()) for j in range(h_kv)], 1)
        kq, vq = kq.view(np.uint8), vq.view(np.uint8)
    else:
        kq, vq = kn.view(torch.uint8).numpy(), vn.view(torch.uint8).numpy()
    # pools viewed as raw bytes: [num_pages, h_kv, 16, d * element bytes]
    oracle.scatter_append(exp_k, slots, kq)
    oracle.scatter_append(exp_v, slots, vq)
    pkv.kv_append(kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    assert pkv.device_error() == 0
    np.testing.assert_array_equal(raw(kc), exp_k)
    np.testing.assert_array_equal(raw(vc), exp_v)


# Scales for the quantiser checks: ordinary ones, significands of all ones and of one, the
# ends of the range where the append divides with a precomputed reciprocal (2^-80, 2^80) and
# beyond it (where it divides per element), and seeded random ones of every exponent between.
QUANT_SCALES = [1.0, 0.0123, 9.5, 37.0, 0.75, 3e-5, 7e4, float(np.float32(2.0) - np.float32(2**-23)),
                2.0 ** -80, 2.0 ** 80, 2.0 ** -90, 2.0 ** 90] + [
    float(np.float32(m) * np.float32(2.0 ** e))
    for m, e in zip(np.random.default_rng(271).uniform(1, 2, 11), range(-20, 21, 4))]


def test_fp8_quantiser_matches_oracle_on_every_bf16_pattern():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits[~torch.isnan(bits)]
    n = (x.numel() // 128) * 128
    x = x[:n].reshape(-1, 1, 128).contiguous()
    kc = torch.zeros(x.shape[0] // 16 + 1, 1, 16, 128, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.arange(x.shape[0], dtype=torch.int64, device="cuda")
    for s in QUANT_SCALES:
        sc = torch.tensor([s], device="cuda")
        pkv.kv_append(x.cuda(), x.cuda(), slots, kc, vc, sc, sc)
        got = kc.reshape(-1, 128)[:x.shape[0]].cpu().numpy()
        ref = oracle.quantize_e4m3(x.float().numpy().reshape(-1, 128), s)
        np.testing.assert_array_equal(got, ref)
    assert pkv.device_error() == 0


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("int8", [False, True])
def test_absmax_scales_bit_exact(dt, int8):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(3000, 8, 128, generator=g) * torch.linspace(0.1, 50, 8)[None, :, None]
    x[:, 5] = 0  # an all-zero head gets scale 1
    x = x.to(torch.bfloat16 if dt == "bf16" else torch.float32)
    got = pkv.kv_absmax_scales(x.cuda(), int8=int8).cpu().numpy()
    ref = oracle.absmax_scales_per_head(x.float().numpy(), 127.0 if int8 else 448.0)
    np.testing.assert_array_equal(got, ref)


def test_int8_quantiser_matches_oracle_on_every_bf16_pattern():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits[torch.isfinite(bits)]
    n = (x.numel() // 128) * 128
    x = x[:n].reshape(-1, 1, 128).contiguous()
    kc = torch.zeros(x.shape[0] // 16 + 1, 1, 16, 128, dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.arange(x.shape[0], dtype=torch.int64, device="cuda")
    for s in QUANT_SCALES:
        sc = torch.tensor([s], device="cuda")
        pkv.kv_append(x.cuda(), x.cuda(), slots, kc, vc, sc, sc)
        got = kc.reshape(-1, 128)[:x.shape[0]].cpu().numpy()
        ref = oracle.quantize_int8(x.float().numpy().reshape(-1, 128), s)
        np.testing.assert_array_equal(got, ref)
    assert pkv.device_error() == 0


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("n_tok", [2048, 4099, 25001])
def test_prompt_sized_append_bit_exact(int8, n_tok):
    # a prompt-sized batch (bf16 rows into an FP8 or INT8 cache): every bf16 pattern, cycled
    # through the rows, a token count that is not a multiple of the kernel's token pairs, eight
    # per-head scales that include both ends of the reciprocal division's range and beyond,
    # padding slots (-1, skipped) and slots in shuffled pages
    h_kv, d = 8, 128
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    pats = bits[torch.isfinite(bits)] if int8 else bits[~torch.isnan(bits)]
    need = n_tok * h_kv * d
    idx = torch.randperm(need, generator=torch.Generator().manual_seed(n_tok)) % pats.numel()
    k = pats[idx].reshape(n_tok, h_kv, d).contiguous()
    v = pats[idx.flip(0)].reshape(n_tok, h_kv, d).contiguous()
    scales = torch.tensor([1.0, 0.0123, 2.0 ** -80, 2.0 ** 80, 2.0 ** -90, 37.0, 3e-5, 7e4])
    pages = n_tok // 16 + 8
    rng = np.random.default_rng(n_tok)
    slots = (rng.permutation(pages)[:, None] * 16 + np.arange(16)[None, :]).ravel()[:n_tok]
    slots = slots.astype(np.int64)
    slots[rng.choice(n_tok, n_tok // 50, replace=False)] = -1
    dt = torch.int8 if int8 else torch.uint8
    kc = torch.full((pages, h_kv, 16, d), 0x55, dtype=torch.uint8).view(dt).cuda()
    vc = kc.clone()
    sc_k, sc_v = scales.cuda(), scales.flip(0).contiguous().cuda()
    pkv.kv_append(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), kc, vc, sc_k, sc_v)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    quant = oracle.quantize_int8 if int8 else oracle.quantize_e4m3
    for pool, x, sc in ((kc, k, scales), (vc, v, scales.flip(0))):
        got = pool.cpu().numpy().view(np.uint8).copy()
        ref = np.full_like(got, 0x55)
        xf = x.float().numpy()
        codes = np.stack([quant(xf[:, j], float(sc[j])) for j in range(h_kv)], 1).view(np.uint8)
        ok = slots >= 0
        ref[slots[ok] // 16, :, slots[ok] % 16, :] = codes[ok]
        np.testing.assert_array_equal(got, ref)


def test_prompt_sized_append_bad_slot():
    # a prompt-sized append reports a slot past the pool and skips that token only
    n, h_kv, d = 3000, 8, 128
    pages = n // 16 + 1
    x = torch.ones(n, h_kv, d, dtype=torch.bfloat16, device="cuda")
    slots = torch.arange(n, dtype=torch.int64)
    slots[1500] = pages * 16 + 5
    kc = torch.zeros(pages, h_kv, 16, d, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    one = torch.ones(h_kv, device="cuda")
    pkv.device_error()
    pkv.kv_append(x, x, slots.cuda(), kc, vc, one, one)
    assert pkv.device_error() & pkv.DEVERR_BAD_SLOT
    code = int(oracle.quantize_e4m3(np.ones(1, np.float32), 1.0)[0])
    flat = kc.permute(0, 2, 1, 3).reshape(pages * 16, h_kv * d).cpu()
    written = (flat == code).all(1)
    assert int(written.sum()) == n - 1 and not bool(written[1500])


# ---- device error word: bad inputs are skipped, never faulted on ---------------------------------

def test_bad_page_id_sets_error_word():
    w = workloads.custom("badpage", 31, 2, 8, 2, 64, "bf16", "bf16", [40, 20])
    sc = Scenario(w)
    sc.append()
    bt = sc.block_tables.clone()
    bt[0, 1] = w.num_pages + 5
    pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, bt, sc.context_lens, w.scale,
                               workspace=sc.workspace)
    assert pkv.device_error() & pkv.DEVERR_BAD_PAGE
    assert pkv.device_error() == 0  # reading clears it


def test_context_longer_than_table_is_cut_and_flagged():
    w = workloads.custom("longctx", 32, 2, 8, 2, 64, "bf16", "bf16", [40, 20])
    sc = Scenario(w)
    sc.append()
    cl = sc.context_lens.clone()
    cl[1] = 16 * sc.block_tables.shape[1] + 100
    pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables, cl, w.scale,
                               workspace=sc.workspace)
    assert pkv.device_error() & pkv.DEVERR_BAD_PAGE


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_bad_slot_sets_error_word(kv):
    # three tokens (an odd count) with the out-of-range slot in the middle: it is reported and
    # skipped, the other two are written
    fp8 = kv == "fp8_e4m3"
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(3, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([0, 4 * 16, 5], dtype=torch.int64, device="cuda")
    one = torch.ones(2, device="cuda") if fp8 else None
    pkv.device_error()
    pkv.kv_append(kn, kn, slots, kc, vc, one, one)
    assert pkv.device_error() & pkv.DEVERR_BAD_SLOT
    want = int(oracle.quantize_e4m3(np.ones(1, np.float32), 1.0)[0]) if fp8 else 1.0
    got = kc.float() if not fp8 else kc.to(torch.int32)
    assert got[0, :, 0].eq(want).all() and got[0, :, 5].eq(want).all()
    assert int(torch.count_nonzero(kc.view(torch.uint8))) == 2 * 2 * 64 * (1 if fp8 else 2)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_host_step_equals_device_step(kv):
    # one packed host->device copy, the fused step, one device->host copy: same output and
    # pool bytes as the fused step on device-resident inputs
    w = workloads.custom("hoststep", 7300, 5, 8, 2, 128, kv, "bf16", [40, 3, 200, 17, 64])
    a = Scenario(w)
    out_a = a.fused_step().clone()
    b = Scenario(w)
    hs = pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                      b.block_tables.shape[1], q_dtype=b.q.dtype, new_dtype=b.k_new.dtype)
    hs.q_host.copy_(b.q.cpu())
    hs.k_new_host.copy_(b.k_new.cpu())
    hs.v_new_host.copy_(b.v_new.cpu())
    hs.block_tables_host.copy_(b.block_tables.cpu())
    hs.context_lens_host.copy_(b.context_lens.cpu())
    ks, vs = b.scales if b.scales else (None, None)
    out_b = hs.step(b.cache.k, b.cache.v, w.scale, k_scales=ks, v_scales=vs,
                    workspace=b.workspace)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert torch.equal(out_a.cpu(), out_b)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert hs.h2d_bytes >= (b.q.numel() + 2 * b.k_new.numel()) * 2


def test_host_step_output_into_pageable_memory():
    # the packed step's output copy lands in pageable host memory as well as in pinned memory:
    # the same bytes
    import ctypes
    w = workloads.custom("hoststep_pageable", 7302, 5, 8, 2, 128, "bf16", "bf16",
                         [40, 3, 200, 17, 64])
    b = Scenario(w)
    hs = pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                      b.block_tables.shape[1])
    hs.q_host.copy_(b.q.cpu())
    hs.k_new_host.copy_(b.k_new.cpu())
    hs.v_new_host.copy_(b.v_new.cpu())
    hs.block_tables_host.copy_(b.block_tables.cpu())
    hs.context_lens_host.copy_(b.context_lens.cpu())
    pinned = hs.step(b.cache.k, b.cache.v, w.scale, workspace=b.workspace)
    torch.cuda.synchronize()  # (out_host holds the output once the stream gets there)
    pinned = pinned.clone()
    pageable = np.full(pinned.numel(), 0x7fc0, dtype=np.uint16)  # NaN until written
    out_dev = torch.full_like(b.q, float("nan"))
    desc = pkv.cache_desc(b.cache.k)
    st = pkv.lib().pkv_paged_decode_step_packed(
        ctypes.c_void_p(hs.host.data_ptr()), ctypes.c_void_p(hs.dev.data_ptr()), w.batch,
        w.num_q_heads, pkv.BF16, pkv.BF16, ctypes.c_void_p(b.cache.k.data_ptr()),
        ctypes.c_void_p(b.cache.v.data_ptr()), ctypes.byref(desc), b.block_tables.shape[1],
        ctypes.c_float(w.scale), None, None, 0, 0, ctypes.c_void_p(out_dev.data_ptr()),
        ctypes.c_void_p(pageable.ctypes.data), ctypes.c_void_p(b.workspace.data_ptr()),
        b.workspace.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pkv.lib().pkv_last_error().decode()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert np.array_equal(pageable, pinned.view(torch.int16).numpy().view(np.uint16).ravel())
    assert torch.equal(out_dev.cpu(), pinned)


def test_host_step_graph_replays_each_steps_inputs():
    # the captured host step re-reads the pinned inputs on every replay: new queries each
    # step give the same bytes as the step made call by call, and differ between steps
    w = workloads.custom("hoststep_graph", 7301, 5, 8, 2, 128, "bf16", "bf16",
                         [40, 3, 700, 17, 64])
    b = Scenario(w)
    steps = [pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                          b.block_tables.shape[1], use_graph=g) for g in (True, False)]
    for hs in steps:
        hs.k_new_host.copy_(b.k_new.cpu())
        hs.v_new_host.copy_(b.v_new.cpu())
        hs.block_tables_host.copy_(b.block_tables.cpu())
        hs.context_lens_host.copy_(b.context_lens.cpu())
    prev = None
    for it in range(3):
        q = torch.randn(b.q.shape, generator=torch.Generator().manual_seed(it)).to(b.q.dtype)
        outs = []
        for hs in steps:
            hs.q_host.copy_(q)
            hs.step(b.cache.k, b.cache.v, w.scale, workspace=b.workspace)
            torch.cuda.synchronize()
            outs.append(hs.out_host.clone())
        assert pkv.device_error() == 0
        assert torch.equal(outs[0], outs[1])
        if prev is not None:
            assert not torch.equal(prev, outs[0])
        prev = outs[0]


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "int8"])
@pytest.mark.parametrize("wpr", [True, False])
def test_short_single_chunk_batches_both_ways(kv, wpr):
    # every request fits one chunk of <= 16 pages: one warp per request (default) or four warps
    # per request; both match the oracle, the step and append-then-decode agree bitwise
    lens = [1, 16, 17, 100, 255, 3, 64, 200, 33, 129]
    w = workloads.custom("wpr", 7500, len(lens), 16, 4, 128, kv, "bf16", lens)
    pkv.decode_set_warp_per_request(wpr)
    try:
        a = Scenario(w)
        out_a = a.step().clone()
        b = Scenario(w)
        out_b = b.fused_step().clone()
        torch.cuda.synchronize()
    finally:
        pkv.decode_set_warp_per_request(True)
    assert pkv.device_error() == 0
    assert torch.equal(out_a, out_b)
    err = _max_err(out_b, oracle_expected(w))
    assert err <= tolerance(w), err
