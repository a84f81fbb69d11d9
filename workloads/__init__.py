"""Seeded synthetic inputs for single-token paged decode attention.

Shared by the tests, the benchmark and the smoke check, and by both sides of every parity
comparison (the CUDA library and the CPU oracle). This module only draws random numbers: it
holds none of the method's arithmetic -- no page accounting, no slot mapping, no attention,
no quantisation. What it returns is plain input: context lengths, key/value/query values per
request in logical (contiguous) order, the order in which physical pages are handed out, and a
seed for the junk bytes that fill unused pool slots.

Shapes and distributions follow the workloads the KV-cache pages describe: Llama-3-8B-shaped
layers (32 query heads over 8 KV heads, head dim 128, KV Cache and PagedAttention page,
"Memory cost" worked examples), Llama-3-70B-shaped layers (64 over 8), 16-token pages
("PagedAttention" section), a 2000-token shared system prompt ("Prefix caching" section), an
FP8 E4M3 cache ("KV cache quantisation" section) and continuous batching ("Continuous
batching" section). Values are N(0, 1) drawn in fp32 from a seeded torch CPU generator, then
cast to the storage dtype.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE_SIZE = 16
BASE_SEED = 271000


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _normal(shape, dtype: str, g: torch.Generator) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if dtype == "f32":
        return x
    return x.to(torch.bfloat16)


@dataclasses.dataclass
class DecodeInputs:
    """One decode step over a batch of requests.

    Request b attends over ``context_lens[b]`` tokens. Its tokens are the first
    ``prefix_len`` rows of ``prefix_k``/``prefix_v`` (a prompt prefix every request
    shares; empty unless ``prefix_len > 0``) followed by rows
    ``offsets[b] .. offsets[b] + context_lens[b] - prefix_len`` of ``k_tokens``/``v_tokens``.
    The last token of every request is the one the step appends before decoding.
    """

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str  # "f32" | "bf16" | "fp8_e4m3" (fp8: values drawn as bf16, quantised downstream)
    q_dtype: str  # "f32" | "bf16"
    context_lens: np.ndarray  # int32 [B]
    offsets: np.ndarray  # int64 [B]
    k_tokens: torch.Tensor  # [rows, h_kv, d]
    v_tokens: torch.Tensor
    q: torch.Tensor  # [B, h_q, d]
    num_pages: int  # physical pool size in pages
    page_order: np.ndarray  # int32 [num_pages]: random permutation, order pages are handed out
    scale: float
    fill_seed: int
    prefix_len: int = 0
    prefix_k: torch.Tensor | None = None
    prefix_v: torch.Tensor | None = None
    window: int = 0  # > 0: the decode attends the last `window` positions ...
    sink: int = 0  # ... and the first `sink` ones ("Sliding window" section)

    def request_tokens(self, b: int):
        """Keys and values of request b in logical order, as [ctx, h_kv, d] CPU tensors."""
        n_own = int(self.context_lens[b]) - self.prefix_len
        o = int(self.offsets[b])
        k = self.k_tokens[o:o + n_own]
        v = self.v_tokens[o:o + n_own]
        if self.prefix_len:
            k = torch.cat([self.prefix_k, k], 0)
            v = torch.cat([self.prefix_v, v], 0)
        return k, v


def _pool_pages(lens, page_size, slack=0.10, extra=0):
    # pool sizing only: enough pages for every request plus the stated slack
    total = sum(-(-int(n) // page_size) for n in lens)
    return int(math.ceil(total * (1.0 + slack))) + extra


def _assemble(name, seed, batch, h_q, h_kv, d, kv_dtype, q_dtype, lens, num_pages,
              prefix_len=0, page_size=PAGE_SIZE):
    g = _gen(seed)
    lens = np.asarray(lens, dtype=np.int32)
    own = lens.astype(np.int64) - prefix_len
    offsets = np.zeros(batch, dtype=np.int64)
    if batch > 1:
        offsets[1:] = np.cumsum(own)[:-1]
    rows = int(own.sum())
    value_dtype = "f32" if kv_dtype == "f32" else "bf16"
    prefix_k = prefix_v = None
    if prefix_len:
        prefix_k = _normal((prefix_len, h_kv, d), value_dtype, g)
        prefix_v = _normal((prefix_len, h_kv, d), value_dtype, g)
    k = _normal((rows, h_kv, d), value_dtype, g)
    v = _normal((rows, h_kv, d), value_dtype, g)
    q = _normal((batch, h_q, d), q_dtype, g)
    order = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    return DecodeInputs(name=name, batch=batch, num_q_heads=h_q, num_kv_heads=h_kv,
                        head_dim=d, page_size=page_size, kv_dtype=kv_dtype, q_dtype=q_dtype,
                        context_lens=lens, offsets=offsets, k_tokens=k, v_tokens=v, q=q,
                        num_pages=int(num_pages), page_order=order, scale=1.0 / math.sqrt(d),
                        fill_seed=seed + 7, prefix_len=prefix_len, prefix_k=prefix_k,
                        prefix_v=prefix_v)


def tiny_ref() -> DecodeInputs:
    """1 layer, batch 2, 4 query / 2 KV heads, d=64, fp32, 16-token pages, pool of 8 pages.

    17 and 33 tokens are cached; the step appends one token to each, so the decode attends
    over 18 and 34 tokens.
    """
    seed = BASE_SEED + 1
    return _assemble("tiny_ref", seed, 2, 4, 2, 64, "f32", "f32", [18, 34], 8)


def llama3_8b_batch64(batch: int = 64) -> DecodeInputs:
    """Llama-3-8B-shaped layer: 32 q / 8 kv heads, d=128, bf16, context U[512, 4096]."""
    seed = BASE_SEED + 2
    g = _gen(seed - 1000)
    lens = torch.randint(512, 4097, (batch,), generator=g).numpy()
    return _assemble("llama3_8b_decode_b%d" % batch, seed, batch, 32, 8, 128, "bf16", "bf16",
                     lens, _pool_pages(lens, PAGE_SIZE))


def llama3_70b_long() -> DecodeInputs:
    """Llama-3-70B-shaped layer: 64 q / 8 kv heads, d=128, bf16, contexts 131072/65536/32768/8191."""
    seed = BASE_SEED + 3
    lens = [131072, 65536, 32768, 8191]
    return _assemble("llama3_70b_long_b4", seed, 4, 64, 8, 128, "bf16", "bf16", lens,
                     _pool_pages(lens, PAGE_SIZE))


def llama3_8b_window(batch: int = 64, window: int = 1024, sink: int = 4) -> DecodeInputs:
    """Llama-3-8B-shaped layer with a sliding window of 1024 positions plus 4 attention sinks
    ("Sliding window" section: StreamingLLM keeps a few first tokens and the last W), contexts
    U[2048, 6144], so a request attends about a quarter of its cache."""
    seed = BASE_SEED + 6
    g = _gen(seed - 1000)
    lens = torch.randint(2048, 6145, (batch,), generator=g).numpy()
    w = _assemble("llama3_8b_window%d_sink%d_b%d" % (window, sink, batch), seed, batch, 32, 8,
                  128, "bf16", "bf16", lens, _pool_pages(lens, PAGE_SIZE))
    w.window, w.sink = window, sink
    return w


@dataclasses.dataclass
class ParallelSampling:
    """Parallel sampling ("KV Cache" glossary: a prompt's blocks shared by the sequences sampled
    from it): ``prompts`` holds the prompts' tokens (request p = prompt p); each prompt is
    forked into ``samples`` sequences, sample s of prompt p being row p * samples + s of the
    first decode step's ``q`` [P*S, h_q, d] and new rows ``k_new``/``v_new`` [P*S, h_kv, d]."""

    prompts: DecodeInputs
    samples: int
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor


def parallel_sampling(n_prompts: int = 16, samples: int = 4) -> ParallelSampling:
    """16 Llama-3-8B-shaped prompts of U[1000, 3000] tokens (a partly filled last page each),
    4 samples each (batch 64)."""
    seed = BASE_SEED + 7
    g = _gen(seed - 1000)
    lens = torch.randint(1000, 3001, (n_prompts,), generator=g).numpy()
    w = _assemble("parallel_sampling_p%d_s%d" % (n_prompts, samples), seed, n_prompts, 32, 8, 128,
                  "bf16", "bf16", lens, _pool_pages(lens, PAGE_SIZE) + 2 * n_prompts * samples)
    n = n_prompts * samples
    return ParallelSampling(prompts=w, samples=samples, q=_normal((n, 32, 128), "bf16", g),
                            k_new=_normal((n, 8, 128), "bf16", g),
                            v_new=_normal((n, 8, 128), "bf16", g))


def prefix_sharing(batch: int = 128, prefix_len: int = 2000) -> DecodeInputs:
    """128 requests sharing a 2000-token prompt prefix, then own suffixes of U[5, 200] tokens."""
    seed = BASE_SEED + 4
    g = _gen(seed - 1000)
    suffix = torch.randint(5, 201, (batch,), generator=g).numpy()
    lens = prefix_len + suffix
    # the shared prefix occupies its pages once; every copy-layout run needs its own copy too
    pages = _pool_pages(list(lens), PAGE_SIZE) + (-(-prefix_len // PAGE_SIZE))
    return _assemble("prefix_sharing_b%d" % batch, seed, batch, 32, 8, 128, "bf16", "bf16", lens,
                     pages, prefix_len=prefix_len)


@dataclasses.dataclass
class PrefixGroupsInputs:
    """A batch where several prompt prefixes are each shared by a set of requests and the
    other requests share nothing ("Prefix caching" section: requests with a common system
    prompt). Request b belongs to prefix ``group_of[b]`` (-1: none); its tokens are the
    ``prefix_lens[g]`` rows of ``prefix_k[g]``/``prefix_v[g]`` followed by rows
    ``offsets[b] ..`` of ``k_tokens``/``v_tokens``; ``context_lens[b]`` counts both. The last
    token of every request is the one the step appends. bf16 values, bf16 queries."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    group_of: np.ndarray  # int32 [B]
    prefix_lens: np.ndarray  # int32 [n_prefixes], whole pages
    prefix_k: list
    prefix_v: list
    context_lens: np.ndarray  # int32 [B]
    offsets: np.ndarray  # int64 [B]
    k_tokens: torch.Tensor
    v_tokens: torch.Tensor
    q: torch.Tensor
    num_pages: int
    page_order: np.ndarray
    scale: float
    fill_seed: int
    kv_dtype: str = "bf16"
    q_dtype: str = "bf16"

    def request_tokens(self, b: int):
        g = int(self.group_of[b])
        n_pre = int(self.prefix_lens[g]) if g >= 0 else 0
        o, n_own = int(self.offsets[b]), int(self.context_lens[b]) - n_pre
        k, v = self.k_tokens[o:o + n_own], self.v_tokens[o:o + n_own]
        if g >= 0:
            k = torch.cat([self.prefix_k[g][:n_pre], k], 0)
            v = torch.cat([self.prefix_v[g][:n_pre], v], 0)
        return k, v


def prefix_groups(name, seed, h_q, h_kv, d, groups, singles=(), slack=0.10):
    """``groups``: (prefix pages, members, lowest, highest own length) per prefix; own lengths
    are U[lowest, highest] (>= 1: the step's token); ``singles``: (lowest, highest) length
    ranges of requests with no shared prefix. Batch order is a seeded shuffle of them all."""
    g = _gen(seed)
    kinds = []
    for gi, (_, members, lo, hi) in enumerate(groups):
        kinds += [(gi, lo, hi)] * int(members)
    kinds += [(-1, lo, hi) for lo, hi in singles]
    perm = torch.randperm(len(kinds), generator=g).tolist()
    kinds = [kinds[i] for i in perm]
    B = len(kinds)
    prefix_lens = np.array([int(p) * PAGE_SIZE for p, _, _, _ in groups], dtype=np.int32)
    group_of = np.array([k[0] for k in kinds], dtype=np.int32)
    own = np.array([int(torch.randint(lo, hi + 1, (1,), generator=g)) for _, lo, hi in kinds],
                   dtype=np.int64)
    lens = own + np.array([prefix_lens[k[0]] if k[0] >= 0 else 0 for k in kinds], dtype=np.int64)
    offsets = np.zeros(B, dtype=np.int64)
    if B > 1:
        offsets[1:] = np.cumsum(own)[:-1]
    pk = [_normal((int(n), h_kv, d), "bf16", g) for n in prefix_lens]
    pv = [_normal((int(n), h_kv, d), "bf16", g) for n in prefix_lens]
    k = _normal((int(own.sum()), h_kv, d), "bf16", g)
    v = _normal((int(own.sum()), h_kv, d), "bf16", g)
    q = _normal((B, h_q, d), "bf16", g)
    pages = _pool_pages(list(own + PAGE_SIZE), PAGE_SIZE, slack) + int(sum(p for p, *_ in groups))
    order = torch.randperm(pages, generator=g).numpy().astype(np.int32)
    return PrefixGroupsInputs(name=name, batch=B, num_q_heads=h_q, num_kv_heads=h_kv, head_dim=d,
                              page_size=PAGE_SIZE, group_of=group_of, prefix_lens=prefix_lens,
                              prefix_k=pk, prefix_v=pv, context_lens=lens.astype(np.int32),
                              offsets=offsets, k_tokens=k, v_tokens=v, q=q, num_pages=int(pages),
                              page_order=order, scale=1.0 / math.sqrt(d), fill_seed=seed + 7)


def custom(name, seed, batch, h_q, h_kv, d, kv_dtype, q_dtype, lens, slack=0.10,
           prefix_len=0) -> DecodeInputs:
    """Any shape, for parity sweeps and edge cases."""
    pages = _pool_pages(lens, PAGE_SIZE, slack) + (-(-prefix_len // PAGE_SIZE)) + 1
    return _assemble(name, seed, batch, h_q, h_kv, d, kv_dtype, q_dtype, lens, pages,
                     prefix_len=prefix_len)


@dataclasses.dataclass
class ContinuousBatchingTrace:
    """Continuous batching over an FP8 E4M3 cache: B request slots, ``steps`` decode steps.

    Slot b starts with request b holding ``initial_lens[b]`` cached tokens. Every step
    appends one token to each live request and decodes. ``finish[s, b]`` says the request in
    slot b finishes after step s; before step s+1 it is replaced by a new request whose prompt
    has ``replacement_lens[s, b]`` tokens. ``rid_table[s, b]`` is the id of the request in slot
    b during step s (0..B-1 for the initial ones, then B, B+1, ... in (step, slot) order).
    """

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    steps: int
    initial_lens: np.ndarray
    finish: np.ndarray  # bool [steps, B]
    replacement_lens: np.ndarray  # int32 [steps, B]
    num_pages: int
    page_order: np.ndarray
    scale: float
    seed: int
    rid_table: np.ndarray = None  # int64 [steps, B]
    prompt_lens: np.ndarray = None  # int32 [number of requests]

    def __post_init__(self):
        B, S = self.batch, self.steps
        table = np.zeros((S, B), dtype=np.int64)
        table[0] = np.arange(B)
        prompts = list(self.initial_lens.astype(np.int64))
        for s in range(1, S):
            table[s] = table[s - 1]
            for b in range(B):
                if self.finish[s - 1, b]:
                    table[s, b] = len(prompts)
                    prompts.append(int(self.replacement_lens[s - 1, b]))
        self.rid_table = table
        self.prompt_lens = np.array(prompts, dtype=np.int32)

    def max_rows(self, request_id: int) -> int:
        """Rows a request can ever hold: its prompt plus one appended token per step."""
        return int(self.prompt_lens[request_id]) + self.steps

    def request_tokens(self, request_id: int):
        """Keys and values of a request, bf16 [max_rows, h_kv, d]; the same on every call."""
        n = self.max_rows(request_id)
        shape = (n, self.num_kv_heads, self.head_dim)
        k = _normal(shape, "bf16", _gen(self.seed * 1000003 + 2 * request_id + 17))
        v = _normal(shape, "bf16", _gen(self.seed * 1000003 + 2 * request_id + 18))
        return k, v

    def step_q(self, step: int) -> torch.Tensor:
        g = _gen(self.seed * 7919 + step)
        return _normal((self.batch, self.num_q_heads, self.head_dim), "bf16", g)


def fp8_continuous_batching(batch=256, steps=32, lo=128, hi=8192, rep_lo=128, rep_hi=2048,
                            p_finish=0.05, h_q=32, h_kv=8, d=128) -> ContinuousBatchingTrace:
    """FP8 E4M3 cache with continuous batching: 256 slots, 32 steps, initial contexts
    U[128, 8192], finish probability 0.05 per step, replacements of U[128, 2048] tokens."""
    seed = BASE_SEED + 5
    g = _gen(seed)
    init = torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int32)
    finish = (torch.rand(steps, batch, generator=g) < p_finish).numpy()
    rep = torch.randint(rep_lo, rep_hi + 1, (steps, batch), generator=g).numpy().astype(np.int32)
    pages = _pool_pages(list(init), PAGE_SIZE) + 3 * batch
    order = torch.randperm(pages, generator=g).numpy().astype(np.int32)
    return ContinuousBatchingTrace("fp8_continuous_batching_b%d" % batch, batch, h_q, h_kv, d,
                                   PAGE_SIZE, steps, init, finish, rep, pages, order,
                                   1.0 / math.sqrt(d), seed)
