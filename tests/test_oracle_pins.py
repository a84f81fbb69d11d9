"""Pins for the CPU oracle: checks against what the KV-cache pages print and what mathematics
or independent libraries fix -- never against the oracle itself. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---- memory formula and page accounting -------------------------------------------------------

def test_memory_formula_worked_examples():
    g = _golden("kv_memory_worked_examples.json")
    for ex in g["per_token"]:
        assert oracle.kv_bytes_per_token(ex["L"], ex["h_kv"], ex["d_h"], ex["b"]) == ex["bytes"]
    for ex in g["per_request"]:
        d_kv = ex["h_kv"] * ex["d_h"]
        assert oracle.total_kv_bytes(ex["B"], ex["T"], ex["L"], d_kv, ex["b"]) == ex["bytes"]
    # the printed approximations: 128 KB, ~1 GB, 320 KB, ~40 GB in binary units
    assert g["per_token"][0]["bytes"] == 128 * 2**10
    assert g["per_request"][0]["bytes"] == 1 * 2**30
    assert g["per_token"][1]["bytes"] == 320 * 2**10
    assert g["per_request"][1]["bytes"] == 40 * 2**30


def test_memory_formula_is_linear_in_each_factor():
    # "the KV cache size scales linearly with the number of layers, heads, and the sequence
    # length" (KV-Cache & Paged Attention, Common mistakes)
    base = oracle.total_kv_bytes(3, 100, 5, 7 * 64, 2)
    assert oracle.total_kv_bytes(6, 100, 5, 7 * 64, 2) == 2 * base
    assert oracle.total_kv_bytes(3, 300, 5, 7 * 64, 2) == 3 * base
    assert oracle.total_kv_bytes(3, 100, 10, 7 * 64, 2) == 2 * base
    assert oracle.total_kv_bytes(3, 100, 5, 14 * 64, 2) == 2 * base


def test_page_accounting_17_tokens():
    for c in _golden("page_accounting.json")["cases"]:
        assert oracle.pages_needed(c["n_tokens"], c["page_size"]) == c["pages"]
        assert oracle.wasted_slots(c["n_tokens"], c["page_size"]) == c["wasted_slots"]
        # the 17 tokens split 16 + 1 over the two pages of a table
        table = [5, 2]
        slots = [oracle.slot_of(table, p, c["page_size"]) for p in range(c["n_tokens"])]
        per_page = [sum(1 for s in slots if s // c["page_size"] == pg) for pg in table]
        assert per_page == c["tokens_per_page"]


@pytest.mark.parametrize("P", [1, 8, 16, 32])
def test_pages_needed_is_smallest_cover(P):
    for n in range(0, 200):
        k = oracle.pages_needed(n, P)
        assert k * P >= n and (k == 0 or (k - 1) * P < n)
        assert 0 <= oracle.wasted_slots(n, P) < P or n == 0


def test_slot_mapping_bijective_and_page_local():
    rng = np.random.default_rng(0)
    P, num_pages = 16, 40
    perm = rng.permutation(num_pages)
    lens = [17, 33, 1, 64]
    tables, used = [], 0
    for n in lens:
        k = oracle.pages_needed(n, P)
        tables.append(list(perm[used:used + k]) + [0] * (5 - k))
        used += k
    bt = np.array(tables, dtype=np.int32)
    seen = set()
    for b, n in enumerate(lens):
        s = oracle.slot_mapping(bt, np.arange(n), P, requests=np.full(n, b))
        for p, slot in enumerate(s):
            assert slot // P == bt[b][p // P] and slot % P == p % P
            assert slot not in seen
            seen.add(int(slot))
    assert oracle.slot_mapping(bt, np.array([-1, 3]), P)[0] == -1


# ---- paging: gather is the naive contiguous cache ---------------------------------------------

def _naive_cache(tokens):
    """The naive cache of the pages' section 3: concatenate each new token along time."""
    cache = None
    for t in range(tokens.shape[0]):
        new = tokens[t:t + 1]
        cache = new if cache is None else np.concatenate([cache, new], axis=0)
    return cache


def test_gather_after_append_equals_naive_concatenation():
    rng = np.random.default_rng(1)
    P, h_kv, d, num_pages = 16, 3, 8, 12
    n = 37
    toks = rng.standard_normal((n, h_kv, d))
    table = rng.permutation(num_pages)[:oracle.pages_needed(n, P)]
    pool = np.full((num_pages, h_kv, P, d), np.nan)
    bt = np.array([table], dtype=np.int32)
    for p in range(n):  # one write phase per token
        s = oracle.slot_mapping(bt, np.array([p]), P)
        oracle.scatter_append(pool, s, toks[p:p + 1], P)
    got = oracle.gather_contiguous(pool, table, n, P)
    np.testing.assert_array_equal(got, _naive_cache(toks))


def _pool_from_tokens(k_tok, v_tok, lens, offsets, order, num_pages, P, fill=np.nan,
                      prefix=None):
    """Lay requests out in a pool with the oracle's own scatter; pages come from ``order``."""
    h_kv, d = k_tok.shape[1], k_tok.shape[2]
    kp = np.full((num_pages, h_kv, P, d), fill)
    vp = np.full((num_pages, h_kv, P, d), fill)
    maxp = max(oracle.pages_needed(int(n), P) for n in lens)
    bt = np.zeros((len(lens), maxp), dtype=np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        k = oracle.pages_needed(int(n), P)
        bt[b, :k] = order[nxt:nxt + k]
        nxt += k
        rows = np.arange(int(n))
        s = oracle.slot_mapping(bt, rows, P, requests=np.full(len(rows), b))
        oracle.scatter_append(kp, s, k_tok[offsets[b]:offsets[b] + n], P)
        oracle.scatter_append(vp, s, v_tok[offsets[b]:offsets[b] + n], P)
    return kp, vp, bt


def test_paged_output_independent_of_physical_placement():
    rng = np.random.default_rng(2)
    B, h_q, h_kv, d, P = 3, 4, 2, 16, 16
    lens = np.array([17, 40, 5], dtype=np.int32)
    offsets = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    K = rng.standard_normal((lens.sum(), h_kv, d))
    V = rng.standard_normal((lens.sum(), h_kv, d))
    q = rng.standard_normal((B, h_q, d)).astype(np.float32)
    num_pages = 12
    outs = []
    for seed in (10, 11, 12):
        order = np.random.default_rng(seed).permutation(num_pages)
        kp, vp, bt = _pool_from_tokens(K.astype(np.float32), V.astype(np.float32), lens,
                                       offsets, order, num_pages, P)
        outs.append(oracle.paged_decode(q, "f32", kp.astype(np.float32), vp.astype(np.float32),
                                        "f32", bt, lens, 0.25))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    ref = oracle.contiguous_decode(q, "f32", K.astype(np.float32), V.astype(np.float32), "f32",
                                   offsets, lens, 0.25)
    np.testing.assert_array_equal(outs[0], ref)


def test_shared_prefix_pages_equal_copied_prefix_pages():
    rng = np.random.default_rng(3)
    B, h_q, h_kv, d, P = 4, 4, 2, 8, 16
    prefix = 32  # two full pages shared by every request
    suffix = np.array([3, 16, 20, 1])
    lens = prefix + suffix
    pk = rng.standard_normal((prefix, h_kv, d)).astype(np.float32)
    pv = rng.standard_normal((prefix, h_kv, d)).astype(np.float32)
    sk = rng.standard_normal((suffix.sum(), h_kv, d)).astype(np.float32)
    sv = rng.standard_normal((suffix.sum(), h_kv, d)).astype(np.float32)
    soff = np.concatenate([[0], np.cumsum(suffix)[:-1]])
    q = rng.standard_normal((B, h_q, d)).astype(np.float32)
    num_pages = 20
    maxp = oracle.pages_needed(int(lens.max()), P)
    # shared: pages 0 and 1 hold the prefix once; every table points at them
    kp = np.full((num_pages, h_kv, P, d), np.nan, dtype=np.float32)
    vp = kp.copy()
    bt_shared = np.zeros((B, maxp), dtype=np.int32)
    bt_shared[:, :2] = [0, 1]
    s = oracle.slot_mapping(bt_shared, np.arange(prefix), P, requests=np.zeros(prefix, int))
    oracle.scatter_append(kp, s, pk, P)
    oracle.scatter_append(vp, s, pv, P)
    nxt = 2
    for b in range(B):
        k = oracle.pages_needed(int(lens[b]), P) - 2
        bt_shared[b, 2:2 + k] = range(nxt, nxt + k)
        nxt += k
        pos = np.arange(prefix, lens[b])
        s = oracle.slot_mapping(bt_shared, pos, P, requests=np.full(len(pos), b))
        oracle.scatter_append(kp, s, sk[soff[b]:soff[b] + suffix[b]], P)
        oracle.scatter_append(vp, s, sv[soff[b]:soff[b] + suffix[b]], P)
    shared = oracle.paged_decode(q, "f32", kp, vp, "f32", bt_shared, lens, 0.3)
    # copied: every request owns a private copy of the prefix
    K = np.concatenate([np.concatenate([pk, sk[soff[b]:soff[b] + suffix[b]]]) for b in range(B)])
    V = np.concatenate([np.concatenate([pv, sv[soff[b]:soff[b] + suffix[b]]]) for b in range(B)])
    off = np.concatenate([[0], np.cumsum(lens)[:-1]])
    kp2, vp2, bt2 = _pool_from_tokens(K, V, lens, off, np.arange(30)[::-1], 30, P)
    copied = oracle.paged_decode(q, "f32", kp2.astype(np.float32), vp2.astype(np.float32), "f32",
                                 bt2, lens, 0.3)
    np.testing.assert_array_equal(shared, copied)


# ---- attention: closed forms, library routine, brute force -------------------------------------

def test_single_token_context_returns_its_value():
    rng = np.random.default_rng(4)
    q, K, V = rng.standard_normal(8), rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    np.testing.assert_array_equal(oracle.attend(q, K, V, 0.7), V[0])


def test_equal_keys_give_mean_value():
    rng = np.random.default_rng(5)
    T, d = 23, 16
    q = rng.standard_normal(d)
    K = np.tile(rng.standard_normal(d), (T, 1))
    V = rng.standard_normal((T, d))
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.5), V.mean(0), rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value():
    T, d = 31, 8
    q = np.zeros(d)
    q[0] = 1.0
    K = np.zeros((T, d))
    K[17, 0] = 1000.0
    V = np.random.default_rng(6).standard_normal((T, d))
    np.testing.assert_allclose(oracle.attend(q, K, V, 1.0), V[17], rtol=0, atol=1e-300)


def test_zero_length_context_gives_zero():
    out = oracle.attend(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    np.testing.assert_array_equal(out, np.zeros(4))


def test_softmax_invariant_to_a_key_shift_along_nothing():
    # adding the same vector c to every key adds scale*<q,c> to every score: no change
    rng = np.random.default_rng(7)
    T, d = 19, 8
    q, K, V = rng.standard_normal(d), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    c = rng.standard_normal(d)
    a = oracle.attend(q, K, V, 0.4)
    b = oracle.attend(q, K + c, V, 0.4)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def _sdpa(q, k, v, scale):
    """torch's scaled_dot_product_attention in float64 on CPU, GQA with consecutive groups."""
    qt = torch.from_numpy(q)[None, :, None, :]  # [1, h_q, 1, d]
    kt = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))[None]  # [1, h_kv, T, d]
    vt = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, scale=scale, enable_gqa=True)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("h_q,h_kv", [(4, 4), (8, 2), (32, 8), (6, 1), (16, 1)])
def test_decode_matches_torch_sdpa(h_q, h_kv):
    rng = np.random.default_rng(8 + h_q + h_kv)
    B, d = 3, 16
    lens = np.array([1, 17, 50], dtype=np.int32)
    off = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    K = rng.standard_normal((lens.sum(), h_kv, d))
    V = rng.standard_normal((lens.sum(), h_kv, d))
    q = rng.standard_normal((B, h_q, d))
    got = oracle.contiguous_decode(q.astype(np.float32), "f32", K.astype(np.float32),
                                   V.astype(np.float32), "f32", off, lens, 0.3)
    for b in range(B):
        ref = _sdpa(q[b].astype(np.float32).astype(np.float64),
                    K[off[b]:off[b] + lens[b]].astype(np.float32).astype(np.float64),
                    V[off[b]:off[b] + lens[b]].astype(np.float32).astype(np.float64), 0.3)
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-12)


def test_wrong_head_grouping_would_fail_the_sdpa_pin():
    # planted mistake: interleaved grouping (h % h_kv) instead of consecutive groups
    rng = np.random.default_rng(9)
    h_q, h_kv, d, T = 8, 2, 8, 12
    q = rng.standard_normal((1, h_q, d)).astype(np.float32)
    K = rng.standard_normal((T, h_kv, d)).astype(np.float32)
    V = rng.standard_normal((T, h_kv, d)).astype(np.float32)
    perm = [(h % h_kv) * (h_q // h_kv) + h // h_kv for h in range(h_q)]
    wrong = oracle.contiguous_decode(q[:, perm], "f32", K, V, "f32", [0], [T], 0.5)[0]
    wrong = wrong[np.argsort(perm)]
    ref = _sdpa(q[0].astype(np.float64), K.astype(np.float64), V.astype(np.float64), 0.5)
    assert np.abs(wrong - ref).max() > 1e-3


def test_bf16_inputs_read_exactly():
    rng = np.random.default_rng(10)
    B, h_q, h_kv, d = 2, 4, 2, 8
    lens = np.array([5, 9], dtype=np.int32)
    off = np.array([0, 5], dtype=np.int64)
    K = torch.from_numpy(rng.standard_normal((14, h_kv, d)).astype(np.float32)).bfloat16()
    V = torch.from_numpy(rng.standard_normal((14, h_kv, d)).astype(np.float32)).bfloat16()
    q = torch.from_numpy(rng.standard_normal((B, h_q, d)).astype(np.float32)).bfloat16()
    a = oracle.contiguous_decode(oracle.as_raw(q, "bf16"), "bf16", oracle.as_raw(K, "bf16"),
                                 oracle.as_raw(V, "bf16"), "bf16", off, lens, 0.5)
    b = oracle.contiguous_decode(q.float().numpy(), "f32", K.float().numpy(), V.float().numpy(),
                                 "f32", off, lens, 0.5)
    np.testing.assert_array_equal(a, b)


def test_brute_force_tiny():
    rng = np.random.default_rng(11)
    T, d = 6, 4
    q, K, V = rng.standard_normal(d), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    x = [0.9 * sum(q[i] * K[t][i] for i in range(d)) for t in range(T)]
    w = [math.exp(v) for v in x]
    ref = [sum(w[t] * V[t][i] for t in range(T)) / sum(w) for i in range(d)]
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.9), ref, rtol=0, atol=1e-13)


def test_tiny_workload_against_sdpa():
    w = workloads.tiny_ref()
    got = oracle.decode_inputs(w)
    for b in range(w.batch):
        k, v = w.request_tokens(b)
        ref = _sdpa(w.q[b].double().numpy(), k.double().numpy(), v.double().numpy(), w.scale)
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-12)


# ---- FP8 E4M3 --------------------------------------------------------------------------------------

def test_e4m3_code_values_from_spec():
    for f in _golden("e4m3_codes.json")["facts"]:
        v = oracle.e4m3_value(f["code"])
        if f["value"] == "nan":
            assert math.isnan(v)
        else:
            assert v == f["value"] and math.copysign(1, v) == math.copysign(1, f["value"])


def test_e4m3_table_monotone_and_round_trips():
    tab = oracle.e4m3_table()
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(tab[0x80:0xFF], -pos)
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(tab[c]) == c


def test_e4m3_ties_to_even_and_saturation():
    enc = oracle.e4m3_encode
    assert enc(1.0625) == 0x38  # between 1.0 (0x38) and 1.125 (0x39): even
    assert enc(1.1875) == 0x3A  # between 1.125 and 1.25: even
    assert enc(1.0625 + 2**-20) == 0x39
    assert enc(2**-10) == 0x00  # half the smallest subnormal: ties to zero
    assert enc(3 * 2**-10) == 0x02  # between 2^-9 (0x01) and 2^-8 (0x02): even
    assert enc(-3 * 2**-10) == 0x82
    for big in (448.0, 449.0, 463.99, 464.0, 1e30, float("inf")):
        assert enc(big) == 0x7E and enc(-big) == 0xFE
    assert enc(-0.0) == 0x80 and enc(-1e-30) == 0x80 and enc(0.0) == 0x00


def _torch_e4m3(y32: torch.Tensor) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn cast (round to nearest even) after clamping to +-448."""
    return y32.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_quantiser_matches_torch_on_every_bf16_pattern():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).float()
    x = x[~torch.isnan(x)]
    for s in (1.0, 0.0123, 3.7e-3, 9.5):
        ref = _torch_e4m3(x / torch.tensor(s, dtype=torch.float32))
        got = oracle.quantize_e4m3(x.numpy(), s)
        np.testing.assert_array_equal(got, ref)


def test_absmax_scale_closed_form():
    x = np.zeros((5, 2, 4), dtype=np.float32)
    x[3, 0, 1] = -7.5
    x[1, 0, 2] = 3.0
    x[0, 1, 0] = 0.0
    s = oracle.absmax_scales_per_head(x)
    assert s[0] == np.float32(7.5) / np.float32(448.0)
    assert s[1] == np.float32(1.0)  # all-zero head
    # the largest magnitude quantises to the largest code
    assert oracle.quantize_e4m3(np.array([-7.5], dtype=np.float32), s[0])[0] == 0xFE


def test_fp8_decode_uses_code_value_times_scale():
    rng = np.random.default_rng(12)
    T, h_kv, d = 9, 2, 8
    codes_k = rng.integers(0, 0x7F, (T, h_kv, d)).astype(np.uint8)
    codes_v = rng.integers(0x80, 0xFF, (T, h_kv, d)).astype(np.uint8)
    ks = np.array([0.5, 2.0], dtype=np.float32)
    vs = np.array([0.25, 4.0], dtype=np.float32)
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    got = oracle.contiguous_decode(q, "f32", codes_k, codes_v, "fp8_e4m3", [0], [T], 0.3, ks, vs)
    tab = oracle.e4m3_table()
    K = tab[codes_k] * ks[None, :, None]
    V = tab[codes_v] * vs[None, :, None]
    ref = _sdpa(q[0].astype(np.float64), K, V, 0.3)
    np.testing.assert_allclose(got[0], ref, rtol=0, atol=1e-12)


# ---- allocator model ----------------------------------------------------------------------------

def test_allocator_model_invariants():
    a = oracle.AllocatorModel(8, initial_order=[3, 1, 4, 0, 5, 2, 6, 7])
    x = a.alloc(3)
    assert x == [3, 1, 4]
    a.incref([1])
    a.decref([1, 3])
    assert a.ref[1] == 1 and a.ref[3] == 0 and a.num_free() == 6
    assert a.alloc(1) == [3]  # LIFO: the page just freed comes back first
    with pytest.raises(MemoryError):
        a.alloc(6)
    assert a.num_free() == 5  # all-or-nothing
    with pytest.raises(ValueError):
        a.decref([0])  # never allocated
    with pytest.raises(ValueError):
        a.decref([4, 4])  # would go below zero
    assert sum(1 for r in a.ref if r > 0) + a.num_free() == a.num_pages


# ---- sliding window and attention sinks ("KV cache and PagedAttention", section 8) -------------

def _window_case(seed, T=40, d=8, h_q=4, h_kv=2):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, h_kv, d)).astype(np.float32)
    V = rng.standard_normal((T, h_kv, d)).astype(np.float32)
    q = rng.standard_normal((1, h_q, d)).astype(np.float32)
    return q, K, V


def test_attended_token_sets():
    assert oracle.attended_tokens(10) == list(range(10))
    assert oracle.attended_tokens(10, window=3) == [7, 8, 9]
    assert oracle.attended_tokens(10, sink=2, window=3) == [0, 1, 7, 8, 9]
    assert oracle.attended_tokens(4, sink=2, window=3) == [0, 1, 2, 3]  # overlap
    assert oracle.attended_tokens(10, sink=4, window=0) == list(range(10))  # no window


def test_window_covering_everything_is_full_attention():
    q, K, V = _window_case(20)
    full = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [40], 0.4)
    wide = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [40], 0.4, window=40)
    wider = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [40], 0.4, sink=5, window=100)
    np.testing.assert_array_equal(full, wide)
    np.testing.assert_array_equal(full, wider)


def test_window_of_one_returns_the_newest_value():
    q, K, V = _window_case(21)
    out = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [40], 0.4, window=1)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], V[39, h // 2].astype(np.float64))


def test_window_and_sinks_match_sdpa_with_a_boolean_mask():
    q, K, V = _window_case(22)
    T, sink, window = 40, 3, 9
    got = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [T], 0.4, sink=sink, window=window)
    mask = torch.zeros(1, 1, 1, T, dtype=torch.bool)
    for t in range(T):
        mask[..., t] = t < sink or t >= T - window
    qt = torch.from_numpy(q.astype(np.float64))[:, :, None, :]
    kt = torch.from_numpy(np.ascontiguousarray(K.astype(np.float64).transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V.astype(np.float64).transpose(1, 0, 2)))[None]
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.4,
                                         enable_gqa=True)[0, :, 0, :].numpy()
    np.testing.assert_allclose(got[0], ref, rtol=0, atol=1e-12)


def test_paged_window_reads_only_attended_pages():
    # pages holding no attended token may be gone (page id -1): the window never reads them
    q, K, V = _window_case(23, T=70)
    P = 16
    kp = np.full((8, 2, P, 8), np.nan, dtype=np.float32)
    vp = kp.copy()
    table = np.array([[4, 6, 1, 3, 0]], dtype=np.int32)
    s = oracle.slot_mapping(table, np.arange(70), P, requests=np.zeros(70, int))
    oracle.scatter_append(kp, s, K, P)
    oracle.scatter_append(vp, s, V, P)
    ref = oracle.paged_decode(q, "f32", kp, vp, "f32", table, [70], 0.4, sink=4, window=20)
    table[0, 1] = -1  # tokens 16..31: outside both the 4 sinks and the last 20
    table[0, 2] = -1  # tokens 32..47: likewise
    got = oracle.paged_decode(q, "f32", kp, vp, "f32", table, [70], 0.4, sink=4, window=20)
    np.testing.assert_array_equal(got, ref)
    cont = oracle.contiguous_decode(q, "f32", K, V, "f32", [0], [70], 0.4, sink=4, window=20)
    np.testing.assert_array_equal(got, cont)


# ---- INT8 ("KV cache and PagedAttention", section 7: "INT8 KV: similar") -------------------------

def test_int8_quantiser_closed_forms():
    x = np.array([0.0, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5, 127.4, 200.0, -1e9, 3.49], np.float32)
    np.testing.assert_array_equal(oracle.quantize_int8(x, 1.0),
                                  np.array([0, 0, 2, 2, 0, -2, 126, 127, 127, -127, 3], np.int8))
    s = oracle.absmax_scale(np.array([-6.35, 2.0], np.float32), 127.0)
    assert s == np.float32(6.35) / np.float32(127.0)
    assert oracle.quantize_int8(np.array([-6.35], np.float32), s)[0] == -127


def test_int8_quantiser_matches_torch_on_every_bf16_pattern():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).float()
    x = x[torch.isfinite(x)]
    for s in (1.0, 0.0123, 37.0):
        y = x / torch.tensor(s, dtype=torch.float32)
        ref = torch.round(y).clamp(-127, 127).to(torch.int8).numpy()  # round half to even
        np.testing.assert_array_equal(oracle.quantize_int8(x.numpy(), s), ref)


def test_int8_decode_uses_code_times_scale():
    rng = np.random.default_rng(30)
    T, h_kv, d = 11, 2, 8
    kc = rng.integers(-127, 128, (T, h_kv, d)).astype(np.int8)
    vc = rng.integers(-127, 128, (T, h_kv, d)).astype(np.int8)
    ks = np.array([0.01, 0.2], np.float32)
    vs = np.array([0.05, 0.003], np.float32)
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    got = oracle.contiguous_decode(q, "f32", kc, vc, "int8", [0], [T], 0.3, ks, vs)
    ref = _sdpa(q[0].astype(np.float64), kc * ks[None, :, None].astype(np.float64),
                vc * vs[None, :, None].astype(np.float64), 0.3)
    np.testing.assert_allclose(got[0], ref, rtol=0, atol=1e-12)
