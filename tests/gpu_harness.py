"""Drives the CUDA library through its public API for a ``workloads.DecodeInputs`` case and
computes the oracle's answer for the same inputs. Used by the GPU tests and the benchmark."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_271_gb300 as pkv
from paged_kv_cache_271_gb300.cache import PagedKVCache

POOL_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
              "int8": torch.int8}
CODED = ("fp8_e4m3", "int8")


def fill_junk(t: torch.Tensor, seed: int):
    """Unused pool slots hold random bytes (NaN and Inf patterns included): stale pages."""
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    raw = t.view(torch.uint8)
    raw.copy_(torch.randint(0, 256, raw.shape, dtype=torch.uint8, device=t.device, generator=g))


class Scenario:
    """A decode step set up through the library: pools filled by kv_append via the host
    allocator and slot mapping, then this step's token appended."""

    def __init__(self, w, device="cuda", share_prefix=True, page_order=None, junk=True):
        self.w = w
        self.device = torch.device(device)
        order = w.page_order if page_order is None else page_order
        self.scales = None
        ks = vs = None
        if w.kv_dtype in CODED:
            k_all, v_all = self.all_token_rows()
            i8 = w.kv_dtype == "int8"
            ks = pkv.kv_absmax_scales(k_all.to(self.device), int8=i8)
            vs = pkv.kv_absmax_scales(v_all.to(self.device), int8=i8)
            self.scales = (ks, vs)
        self.cache = PagedKVCache(w.num_pages, w.num_kv_heads, w.head_dim,
                                  POOL_DTYPE[w.kv_dtype], self.device,
                                  initial_free_order=order, k_scales=ks, v_scales=vs)
        if junk:
            fill_junk(self.cache.k, w.fill_seed)
            fill_junk(self.cache.v, w.fill_seed + 1)
        self.rids = list(range(w.batch))
        P = w.page_size
        shared = bool(w.prefix_len and share_prefix)
        if shared:
            owner = -1
            self.cache.add_request(owner)
            s = self.cache.reserve([owner], [w.prefix_len])
            self.cache.write(s, w.prefix_k.to(self.device), w.prefix_v.to(self.device))
            pages = self.cache.pages[owner][:w.prefix_len // P]
            for b in self.rids:
                self.cache.add_request(b, shared_pages=pages, shared_len=w.prefix_len)
            self.cache.free_request(owner)
            self.shared_pages = list(pages)
        else:
            for b in self.rids:
                self.cache.add_request(b)
            self.shared_pages = []
        # prefill everything except each request's last token
        skip = w.prefix_len if shared else 0
        counts = [int(n) - 1 - skip for n in w.context_lens]
        rows_k, rows_v = [], []
        for b in self.rids:
            k, v = w.request_tokens(b)
            rows_k.append(k[skip:skip + counts[b]])
            rows_v.append(v[skip:skip + counts[b]])
        if sum(counts):
            s = self.cache.reserve(self.rids, counts)
            self.cache.write(s, torch.cat(rows_k, 0).to(self.device),
                             torch.cat(rows_v, 0).to(self.device))
        # this step: append the newest token of every request
        self.step_slots = self.cache.reserve(self.rids, [1] * w.batch)
        self.k_new = torch.stack([w.request_tokens(b)[0][-1] for b in self.rids]).to(self.device)
        self.v_new = torch.stack([w.request_tokens(b)[1][-1] for b in self.rids]).to(self.device)
        self.slots_dev = torch.from_numpy(self.step_slots).to(self.device)
        self.q = w.q.to(self.device)
        self.block_tables = torch.from_numpy(self.cache.block_table_array(self.rids)).to(self.device)
        self.context_lens = torch.from_numpy(self.cache.context_lens_array(self.rids)).to(self.device)
        self.out = torch.empty_like(self.q)
        maxp = self.block_tables.shape[1]
        need = pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, maxp)
        self.workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=self.device)

    def all_token_rows(self):
        """Every K and V row of the workload (prefix once), the set the FP8 scales cover."""
        w = self.w
        ks, vs = [w.k_tokens], [w.v_tokens]
        if w.prefix_len:
            ks.insert(0, w.prefix_k)
            vs.insert(0, w.prefix_v)
        return torch.cat(ks, 0), torch.cat(vs, 0)

    def append(self, stream=None):
        self.cache.write(self.slots_dev, self.k_new, self.v_new, stream)

    def decode(self, stream=None):
        ks, vs = self.scales if self.scales else (None, None)
        return pkv.paged_decode_attention(self.q, self.cache.k, self.cache.v, self.block_tables,
                                          self.context_lens, self.w.scale, out=self.out,
                                          k_scales=ks, v_scales=vs, workspace=self.workspace,
                                          stream=stream)

    def step(self, stream=None):
        self.append(stream)
        return self.decode(stream)

    def fused_step(self, stream=None, window=0, sink_tokens=0):
        """Append + decode in one launch (pkv_paged_decode_step[_window])."""
        ks, vs = self.scales if self.scales else (None, None)
        return pkv.paged_decode_step(self.q, self.k_new, self.v_new, self.cache.k, self.cache.v,
                                     self.block_tables, self.context_lens, self.w.scale,
                                     out=self.out, k_scales=ks, v_scales=vs,
                                     workspace=self.workspace, stream=stream, window=window,
                                     sink_tokens=sink_tokens)

    def refresh_tables(self):
        """Re-upload the page tables (after pages were released)."""
        self.block_tables = torch.from_numpy(
            self.cache.block_table_array(self.rids, self.block_tables.shape[1])).to(self.device)


def oracle_fp8_codes(w):
    """The oracle's own per-head scales and codes (E4M3 or INT8) for a quantised workload."""
    kf = w.k_tokens.float().numpy()
    vf = w.v_tokens.float().numpy()
    qmax, quant = (127.0, oracle.quantize_int8) if w.kv_dtype == "int8" else \
        (448.0, oracle.quantize_e4m3)
    ks = oracle.absmax_scales_per_head(kf, qmax)
    vs = oracle.absmax_scales_per_head(vf, qmax)
    kc = np.stack([quant(kf[:, j], ks[j]) for j in range(kf.shape[1])], 1)
    vc = np.stack([quant(vf[:, j], vs[j]) for j in range(vf.shape[1])], 1)
    return ks, vs, kc, vc


def oracle_expected(w, pairs=None, n_threads=0, sink=0, window=0):
    """The oracle's decode output for w, from its own contiguous tokens (and, for FP8, its own
    scales and quantiser). float64 [B, h_q, d] or [n_pairs, d]."""
    if w.kv_dtype not in CODED:
        return oracle.decode_inputs(w, pairs=pairs, n_threads=n_threads, sink=sink, window=window)
    ks, vs, kc, vc = oracle_fp8_codes(w)
    return oracle.decode_inputs(w, pairs=pairs, n_threads=n_threads, k_scales=ks, v_scales=vs,
                                k_codes=kc, v_codes=vc, sink=sink, window=window)


def tolerance(w) -> float:
    """Max-abs bound for the attention output: 1e-5 for fp32 inputs, 1e-2 otherwise."""
    return 1e-5 if w.kv_dtype == "f32" and w.q_dtype == "f32" else 1e-2


class ContinuousBatchingRun:
    """Drives a ``workloads.ContinuousBatchingTrace`` through the library on an FP8 (or, with
    cache_dtype="int8", an INT8) cache: absmax scales over the initial cache, quantising
    prefill of every prompt, one appended token per live request per step, finished requests
    freed and replaced (continuous batching), paged decode every step."""

    def __init__(self, trace, device="cuda", cache_dtype="fp8_e4m3"):
        self.t = trace
        self.device = torch.device(device)
        self.cache_dtype = cache_dtype
        i8 = cache_dtype == "int8"
        B = trace.batch
        self.tokens = {}  # rid -> (k, v) bf16 CPU rows
        for b in range(B):
            self.tokens[b] = trace.request_tokens(b)
        init = [int(n) for n in trace.initial_lens]
        k0 = torch.cat([self.tokens[b][0][:init[b]] for b in range(B)], 0).to(self.device)
        v0 = torch.cat([self.tokens[b][1][:init[b]] for b in range(B)], 0).to(self.device)
        self.k_scales = pkv.kv_absmax_scales(k0, int8=i8)
        self.v_scales = pkv.kv_absmax_scales(v0, int8=i8)
        self.cache = PagedKVCache(trace.num_pages, trace.num_kv_heads, trace.head_dim,
                                  POOL_DTYPE[cache_dtype], self.device,
                                  initial_free_order=trace.page_order,
                                  k_scales=self.k_scales, v_scales=self.v_scales)
        fill_junk(self.cache.k, trace.seed + 11)
        fill_junk(self.cache.v, trace.seed + 12)
        self.slot_rid = list(range(B))
        for b in range(B):
            self.cache.add_request(b)
        slots = self.cache.reserve(self.slot_rid, init)
        self.cache.write(slots, k0, v0)
        del k0, v0
        self.step_index = 0
        self.last_slots = None

    def initial_rows(self):
        """float32 [sum initial, h_kv, d] K and V rows the scales cover (for the oracle)."""
        B = self.t.batch
        init = [int(n) for n in self.t.initial_lens]
        k = torch.cat([self.tokens[b][0][:init[b]] for b in range(B)], 0).float().numpy()
        v = torch.cat([self.tokens[b][1][:init[b]] for b in range(B)], 0).float().numpy()
        return k, v

    def step(self):
        """One continuous-batching step; returns the decode output [B, h_q, d] (bf16)."""
        t, s = self.t, self.step_index
        if s > 0:
            new_rids, counts = [], []
            for b in range(t.batch):
                if t.finish[s - 1, b]:
                    old = self.slot_rid[b]
                    self.cache.free_request(old)
                    del self.tokens[old]
                    rid = int(t.rid_table[s, b])
                    self.slot_rid[b] = rid
                    self.tokens[rid] = t.request_tokens(rid)
                    self.cache.add_request(rid)
                    new_rids.append(rid)
                    counts.append(int(t.prompt_lens[rid]))
            if new_rids:
                slots = self.cache.reserve(new_rids, counts)
                k = torch.cat([self.tokens[r][0][:n] for r, n in zip(new_rids, counts)], 0)
                v = torch.cat([self.tokens[r][1][:n] for r, n in zip(new_rids, counts)], 0)
                self.cache.write(slots, k.to(self.device), v.to(self.device))
        rids = self.slot_rid
        pos = [self.cache.lens[r] for r in rids]
        k_new = torch.stack([self.tokens[r][0][p] for r, p in zip(rids, pos)]).to(self.device)
        v_new = torch.stack([self.tokens[r][1][p] for r, p in zip(rids, pos)]).to(self.device)
        self.last_slots = self.cache.reserve(rids, [1] * len(rids))
        self.cache.write(self.last_slots, k_new, v_new)
        self.k_new, self.v_new = k_new, v_new
        self.q = t.step_q(s).to(self.device)
        self.block_tables = torch.from_numpy(self.cache.block_table_array(rids)).to(self.device)
        self.context_lens = torch.from_numpy(self.cache.context_lens_array(rids)).to(self.device)
        out = pkv.paged_decode_attention(self.q, self.cache.k, self.cache.v, self.block_tables,
                                         self.context_lens, t.scale, k_scales=self.k_scales,
                                         v_scales=self.v_scales)
        self.step_index += 1
        return out

    def oracle_pairs(self, pairs, k_scales, v_scales):
        """Oracle output for (slot, head) pairs of the step just run, from the requests' own
        bf16 rows quantised by the oracle with the given (oracle-computed) scales."""
        t = self.t
        G = t.num_q_heads // t.num_kv_heads
        q = self.q.cpu()
        rows = []
        for b, h in pairs:
            rid = self.slot_rid[b]
            T = self.cache.lens[rid]
            j = h // G
            k = self.tokens[rid][0][:T, j].float().numpy()
            v = self.tokens[rid][1][:T, j].float().numpy()
            quant = oracle.quantize_int8 if self.cache_dtype == "int8" else oracle.quantize_e4m3
            kc = quant(k, k_scales[j])[:, None, :]
            vc = quant(v, v_scales[j])[:, None, :]
            out = oracle.contiguous_decode(oracle.as_raw(q[b:b + 1, h:h + 1], "bf16"), "bf16",
                                           kc, vc, self.cache_dtype, [0], [T], t.scale,
                                           k_scales=k_scales[j:j + 1],
                                           v_scales=v_scales[j:j + 1])
            rows.append(out[0, 0])
        return np.stack(rows)


class GroupScenario:
    """A decode step over a ``workloads.PrefixGroupsInputs`` batch set up through the library:
    each prefix written once and shared (reference counts) by its members' page tables, every
    request's own tokens but the last prefilled, then the step's slots reserved."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.device = torch.device(device)
        P = w.page_size
        self.cache = PagedKVCache(w.num_pages, w.num_kv_heads, w.head_dim, torch.bfloat16,
                                  self.device, initial_free_order=w.page_order)
        fill_junk(self.cache.k, w.fill_seed)
        fill_junk(self.cache.v, w.fill_seed + 1)
        self.rids = list(range(w.batch))
        shared = []
        for g, n in enumerate(w.prefix_lens):
            owner = -1 - g
            self.cache.add_request(owner)
            s = self.cache.reserve([owner], [int(n)])
            self.cache.write(s, w.prefix_k[g].to(self.device), w.prefix_v[g].to(self.device))
            shared.append(list(self.cache.pages[owner][:int(n) // P]))
        for b in self.rids:
            g = int(w.group_of[b])
            if g >= 0:
                self.cache.add_request(b, shared_pages=shared[g], shared_len=int(w.prefix_lens[g]))
            else:
                self.cache.add_request(b)
        for g in range(len(w.prefix_lens)):
            self.cache.free_request(-1 - g)
        self.shared_pages = shared
        pre = [int(w.prefix_lens[w.group_of[b]]) if w.group_of[b] >= 0 else 0 for b in self.rids]
        counts = [int(w.context_lens[b]) - 1 - pre[b] for b in self.rids]
        if sum(counts):
            ks, vs = [], []
            for b in self.rids:
                k, v = w.request_tokens(b)
                ks.append(k[pre[b]:pre[b] + counts[b]])
                vs.append(v[pre[b]:pre[b] + counts[b]])
            s = self.cache.reserve(self.rids, counts)
            self.cache.write(s, torch.cat(ks, 0).to(self.device), torch.cat(vs, 0).to(self.device))
        self.step_slots = self.cache.reserve(self.rids, [1] * w.batch)
        self.slots_dev = torch.from_numpy(self.step_slots).to(self.device)
        self.k_new = torch.stack([w.request_tokens(b)[0][-1] for b in self.rids]).to(self.device)
        self.v_new = torch.stack([w.request_tokens(b)[1][-1] for b in self.rids]).to(self.device)
        self.q = w.q.to(self.device)
        self.bt_host = self.cache.block_table_array(self.rids)
        self.cl_host = self.cache.context_lens_array(self.rids)
        self.block_tables = torch.from_numpy(self.bt_host).to(self.device)
        self.context_lens = torch.from_numpy(self.cl_host).to(self.device)

    def append(self):
        self.cache.write(self.slots_dev, self.k_new, self.v_new)


def oracle_groups_expected(w, pairs=None, n_threads=0):
    """The oracle's decode output for a ``PrefixGroupsInputs`` batch, from each request's own
    contiguous tokens (its prefix followed by its own rows)."""
    ks, vs, offs = [], [], []
    o = 0
    for b in range(w.batch):
        k, v = w.request_tokens(b)
        ks.append(k)
        vs.append(v)
        offs.append(o)
        o += k.shape[0]
    kr = oracle.as_raw(torch.cat(ks, 0), "bf16")
    vr = oracle.as_raw(torch.cat(vs, 0), "bf16")
    return oracle.contiguous_decode(oracle.as_raw(w.q, "bf16"), "bf16", kr, vr, "bf16",
                                    np.array(offs, dtype=np.int64), w.context_lens, w.scale,
                                    pairs=pairs, n_threads=n_threads)
