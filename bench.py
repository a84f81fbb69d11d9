"""Benchmark: one decode step of a Llama-3-8B-shaped layer at batch 64 over a paged KV cache.

A step is the whole hot path for one batch: the host computes this step's slots (page
accounting, slot mapping), then one ``paged_decode_step`` launch writes the new token of each
request into its page (the append) and attends each request's query over its whole cached
context; a combine launch merges the sequences split over several CTAs. Inputs are seeded
synthetic tensors (N(0, 1) bf16, context lengths U[512, 4096]) already resident in HBM. No
step finds its inputs in the L2: identical copies of the KV pools are used in turn (``--l2
rotate``, the default), or the L2 is flushed with a 256 MiB write before every timed step
(``--l2 flush``).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--l2 rotate|flush] [--no-cpu-baseline]

The default workload is the layer above; the others (``--workload``) are the 70B long-context
layer, prefix sharing (plain and cascade), FP8 and INT8 continuous batching (one step's state,
or the whole trace step by step with its frees, replacements and prompt prefills), the prompt
prefill of replacement requests through the quantising append alone (FP8 or INT8 codes), the
sliding window with sinks and the copy-on-write fork of parallel sampling, each measured the
same way.

Prints one JSON line on rank 0. ``value`` is algorithmic HBM bytes per step (K and V of every
attended token, the queries, the outputs, and the appended rows) over the step time, summed
over ranks (replicas: every rank runs its own batch; no collective on the data path).
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = ("paged-decode achieved HBM GB/s (% of GB300 peak) and decode tokens/s at batch 64")
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20


def peaks(kind="hbm_gbs"):
    """A measured peak from MEASURED_PEAKS.json (hbm_gbs, bf16_tflops, ...), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p[kind]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAKS[kind], "fallback"


WORKLOADS = ("llama3_8b_b64", "llama3_70b_long", "prefix_sharing", "prefix_sharing_cascade",
             "fp8_cb_b256", "fp8_cb_b64", "int8_cb_b256", "llama3_8b_window",
             "parallel_sampling_fork", "fp8_cb_trace", "int8_cb_trace", "fp8_prompt_append",
             "int8_prompt_append")


def workload(name="llama3_8b_b64"):
    import workloads
    return {"llama3_8b_b64": workloads.llama3_8b_batch64,
            "llama3_70b_long": workloads.llama3_70b_long,
            "prefix_sharing": workloads.prefix_sharing,
            "prefix_sharing_cascade": workloads.prefix_sharing,
            "llama3_8b_window": workloads.llama3_8b_window}[name]()


def config_of(w):
    return {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
            "kv_dtype": w.kv_dtype, "context_lens": "sum %d" % int(np.sum(w.context_lens)),
            "pool_pages": w.num_pages,
            "l2": "flushed with a 256 MiB write before every timed step",
            "step": DEVICE_STEP}


# What the timed region of a step holds (the host slot mapping runs before it, timed apart).
DEVICE_STEP = ("device: paged_decode_step (append + attention, one launch) + combine, replayed "
               "from a CUDA graph; the host slot mapping is timed apart (host_slot_mapping_us)")


class StepState:
    """Device state of one decode step of a workload, built through the library: the pools
    filled by kv_append, this step's queries and new K/V rows, page tables, context lengths."""

    def __init__(self, name, dev):
        import torch
        import paged_kv_cache_271_gb300 as pkv
        from gpu_harness import ContinuousBatchingRun, Scenario
        self.name = name
        if name.startswith(("fp8_cb", "int8_cb")):
            import workloads
            batch = 64 if name.endswith("_b64") else 256
            coded = "int8" if name.startswith("int8") else "fp8_e4m3"
            tr = workloads.fp8_continuous_batching(batch=batch, steps=4)
            run = ContinuousBatchingRun(tr, device=dev, cache_dtype=coded)
            run.step()
            self.run = run
            self.q, self.k_new, self.v_new = run.q, run.k_new, run.v_new
            self.k, self.v = run.cache.k, run.cache.v
            self.bt, self.cl = run.block_tables, run.context_lens
            self.scales = (run.k_scales, run.v_scales)
            self.scale = tr.scale
            self.batch, self.h_q, self.h_kv, self.d = tr.batch, tr.num_q_heads, tr.num_kv_heads, 128
            self.kv_bytes, self.in_bytes = 1, 2
            self.ctx_sum = int(self.cl.sum())
            wname = tr.name if coded != "int8" else tr.name.replace("fp8", "int8")
            self.config = {"workload": wname + "_state_after_1_step", "batch": tr.batch,
                           "num_q_heads": tr.num_q_heads, "num_kv_heads": tr.num_kv_heads,
                           "head_dim": 128, "page_size": 16, "kv_dtype": coded,
                           "context_lens": "U[128,8192] seeded, sum %d" % self.ctx_sum,
                           "step": DEVICE_STEP}
            self.cache = run.cache
            self.slots = run.last_slots
        else:
            w = workload(name)
            sc = Scenario(w, device=dev)
            self.sc = sc
            self.q, self.k_new, self.v_new = sc.q, sc.k_new, sc.v_new
            self.k, self.v = sc.cache.k, sc.cache.v
            self.bt, self.cl = sc.block_tables, sc.context_lens
            self.scales = sc.scales
            self.scale = w.scale
            self.batch, self.h_q, self.h_kv, self.d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
            self.kv_bytes = {"f32": 4, "bf16": 2, "fp8_e4m3": 1}[w.kv_dtype]
            self.in_bytes = 4 if w.kv_dtype == "f32" else 2
            self.ctx_sum = int(np.sum(w.context_lens))
            self.config = config_of(w)
            self.cache = sc.cache
            self.slots = sc.step_slots
            self.window, self.sink = w.window, w.sink
            if w.window:
                # pages wholly outside every request's window go back to the allocator (their
                # table entries become -1): the step can only read attended pages
                import oracle
                for b in sc.rids:
                    sc.cache.release_outside_window(b, w.window, w.sink)
                sc.refresh_tables()
                self.bt = sc.block_tables
                self.ctx_sum = int(sum(len(oracle.attended_tokens(int(n), w.sink, w.window))
                                       for n in w.context_lens))  # attended tokens
                self.config.update({"window": w.window, "sink_tokens": w.sink,
                                    "attended_tokens": self.ctx_sum})
        self.out = torch.empty_like(self.q)
        self.groups = None
        if name.endswith("_cascade"):
            # the shared prompt's pages computed once per group (pkv_cascade_decode_step)
            self.groups = pkv.cascade_groups(self.bt.cpu().numpy(), self.cl.cpu().numpy())
            self.groups.to(dev)
            g = self.groups
            self.config["step"] = ("device: cascade_decode_step (shared-prefix kernel, append + "
                                   "own-page attention, combine), replayed from a CUDA graph; "
                                   "the host slot mapping and grouping are timed apart "
                                   "(host_slot_mapping_us)")
            self.config["cascade"] = "%d group(s), %s shared pages, %d members max" % (
                g.n_groups, "/".join(str(int(x)) for x in g.prefix_pages), g.max_members)
            need = pkv.cascade_workspace_size(self.batch, self.h_q, self.h_kv, self.d,
                                              self.bt.shape[1], g)
        else:
            need = pkv.decode_workspace_size(self.batch, self.h_q, self.h_kv, self.d,
                                             self.bt.shape[1])
        self.workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)

    def split_label(self):
        """Which split the decode of this step used (autotuning records it on the first call)."""
        import paged_kv_cache_271_gb300 as pkv
        if self.groups is not None and self.groups.n_groups > 0:
            return "cascade (chunks)"
        kv = self.k.dtype
        choice = pkv.decode_split_choice(kv, self.q.dtype, self.batch, self.h_q, self.h_kv,
                                         self.bt.shape[1], getattr(self, "window", 0) or 0,
                                         getattr(self, "sink", 0) or 0, fused=True)
        return {0: "chunks (measured fastest)", 1: "balanced (measured fastest)",
                2: "chunks-x1.5 (1.5 times longer chunks, measured fastest)",
                3: "chunks-x2 (2 times longer chunks, measured fastest)"}.get(
            choice, "chunks (no split measured: one pass or chunks only)")

    def decode_bytes(self):
        """K and V of every attended token + queries + outputs."""
        return self.ctx_sum * self.h_kv * self.d * self.kv_bytes * 2 + 2 * self.batch * self.h_q * self.d * 2

    def append_bytes(self):
        return 2 * self.batch * self.h_kv * self.d * (self.in_bytes + self.kv_bytes)

    def host_step(self):
        """Host part of the step: this step's slots from the page tables (checked)."""
        import paged_kv_cache_271_gb300 as pkv
        bt = self.bt.cpu().numpy() if not hasattr(self, "_bt_host") else self._bt_host
        self._bt_host = bt
        cl = self.cl.cpu().numpy() if not hasattr(self, "_cl_host") else self._cl_host
        self._cl_host = cl
        slots = pkv.slot_mapping(bt, cl.astype(np.int64) - 1, self.cache.num_pages)
        assert np.array_equal(slots, self.slots)
        if self.groups is not None:  # the cascade's groups come from the same host tables
            g = pkv.cascade_groups(bt, cl)
            assert g.n_groups == self.groups.n_groups

    def shared_rows_tokens(self):
        """(query rows, shared tokens) pairs of the cascade groups: every member's query heads
        attend over its group's shared tokens in the prefix kernel."""
        g = self.groups
        return [((int(g.group_offsets[i + 1]) - int(g.group_offsets[i])) * self.h_q,
                 16 * int(g.prefix_pages[i])) for i in range(g.n_groups)]

    def kernel_work(self):
        """Algorithmic work per launch of the step's main kernels: name -> (bound, amount)
        with bytes for HBM-bound kernels and FLOPs for tensor-core ones."""
        if self.groups is None:  # the decode kernel, which also appends the new rows
            return {"paged_decode": ("hbm", self.decode_bytes() + self.append_bytes())}
        row_bytes = self.h_kv * self.d * self.kv_bytes * 2  # K and V of one token
        shared = self.shared_rows_tokens()
        g = self.groups
        # the prefix kernel reads each group's shared pages once and every member's queries
        pre_bytes = (sum(16 * int(p) for p in g.prefix_pages) * row_bytes
                     + sum(r for r, _ in shared) * self.d * 2)
        pre_flops = sum(4.0 * r * t * self.d for r, t in shared)  # Q.K^T and P.V
        own_tokens = self.ctx_sum - sum(t * r // self.h_q for r, t in shared)
        own = own_tokens * row_bytes + 2 * self.batch * self.h_q * self.d * 2 + self.append_bytes()
        return {"cascade_prefix": ("tensor", pre_flops, pre_bytes), "paged_decode": ("hbm", own)}

    def unique_bytes(self):
        """Bytes of distinct pages the step reads (shared pages once) + queries + outputs."""
        bt = self.bt.cpu().numpy()
        cl = self.cl.cpu().numpy()
        pages = set()
        for b in range(self.batch):
            pages.update(int(p) for p in bt[b, :(int(cl[b]) + 15) // 16] if p >= 0)
        tile = 2 * self.h_kv * 16 * self.d * self.kv_bytes
        return len(pages) * tile + 2 * self.batch * self.h_q * self.d * 2

    def used_kv_bytes(self):
        """Bytes of the pool pages that hold tokens (K and V)."""
        a = self.cache.allocator
        used = self.cache.num_pages - a.num_free()
        return used * 2 * self.h_kv * 16 * self.d * self.kv_bytes

    def make_copies(self, n):
        """n identical copies of the K/V pools for steps to use in turn."""
        self.pools = [(self.k, self.v)] + [(self.k.clone(), self.v.clone()) for _ in range(n - 1)]

    def step_call(self, q, k_new, v_new, bt, cl, groups=None, stream=None, pool=0):
        import paged_kv_cache_271_gb300 as pkv
        ks, vs = self.scales if self.scales else (None, None)
        k, v = self.pools[pool] if hasattr(self, "pools") else (self.k, self.v)
        if self.groups is not None:
            return pkv.cascade_decode_step(q, k_new, v_new, k, v, bt, cl, self.scale,
                                           groups or self.groups, out=self.out,
                                           workspace=self.workspace, stream=stream)
        return pkv.paged_decode_step(q, k_new, v_new, k, v, bt, cl, self.scale,
                                     out=self.out, k_scales=ks, v_scales=vs,
                                     workspace=self.workspace, stream=stream,
                                     window=getattr(self, "window", 0),
                                     sink_tokens=getattr(self, "sink", 0))

    def fused_step(self, stream=None, pool=0):
        return self.step_call(self.q, self.k_new, self.v_new, self.bt, self.cl, stream=stream,
                              pool=pool)


# ---- ranks -------------------------------------------------------------------------------------

def rank_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(world_size, backend):
    import torch.distributed as dist
    if world_size > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_rank_step: float, max_ms_per_step: float, world_size: int) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_rank_step * world_size / (max_ms_per_step * 1e-3) / 1e9


# ---- clocks --------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- CPU baseline (the oracle, as it stands) ----------------------------------------------------

def oracle_sample(w, n_seq: int, n_threads: int = 0):
    """Time the fp64 oracle's paged decode on the first n_seq requests of w (all heads), with a
    host pool laid out by the oracle's own allocator model, slot mapping and scatter."""
    import oracle
    P = w.page_size
    alloc = oracle.AllocatorModel(w.num_pages, w.page_order)
    tables, lens = [], []
    for b in range(n_seq):
        tables.append(alloc.alloc(oracle.pages_needed(int(w.context_lens[b]), P)))
        lens.append(int(w.context_lens[b]))
    width = max(len(t) for t in tables)
    bt = np.zeros((n_seq, width), dtype=np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
    used = sorted({p for t in tables for p in t})
    remap = {p: i for i, p in enumerate(used)}  # compact host pool holding only these pages
    bt_c = np.vectorize(lambda p: remap.get(int(p), 0))(bt).astype(np.int32)
    dt = np.uint16 if w.kv_dtype == "bf16" else np.float32
    kp = np.zeros((len(used), w.num_kv_heads, P, w.head_dim), dtype=dt)
    vp = np.zeros_like(kp)
    for b in range(n_seq):
        k, v = w.request_tokens(b)
        slots = oracle.slot_mapping(bt_c, np.arange(lens[b]), P, requests=np.full(lens[b], b))
        oracle.scatter_append(kp, slots, oracle.as_raw(k, w.kv_dtype))
        oracle.scatter_append(vp, slots, oracle.as_raw(v, w.kv_dtype))
    q = oracle.as_raw(w.q[:n_seq], w.q_dtype)
    t0 = time.perf_counter()
    oracle.paged_decode(q, w.q_dtype, kp, vp, w.kv_dtype, bt_c, np.array(lens, dtype=np.int32),
                        w.scale, n_threads=n_threads)
    dt_s = time.perf_counter() - t0
    kvb = {"f32": 4, "bf16": 2}[w.kv_dtype]
    qb = {"f32": 4, "bf16": 2}[w.q_dtype]
    byts = (sum(lens) * w.num_kv_heads * w.head_dim * kvb * 2
            + 2 * n_seq * w.num_q_heads * w.head_dim * qb)
    return byts, dt_s


def cpu_baseline(w, budget_s=12.0):
    import oracle
    threads = oracle.max_threads()
    b1, t1 = oracle_sample(w, 1)
    n = int(min(w.batch, max(1, budget_s / max(t1, 1e-3))))
    byts, t = oracle_sample(w, n) if n > 1 else (b1, t1)
    bs, ts = oracle_sample(w, 1, n_threads=1)
    return {"value": byts / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "fp64 C oracle (gather through page tables + textbook softmax), first %d "
                      "of %d requests, all 32 heads, %.1f s" % (n, w.batch, t),
            "single_thread": {"value": bs / ts / 1e9, "unit": "GB/s",
                              "sample": "first request, all heads, 1 thread, %.2f s" % ts},
            "cpu": _cpu_model()}


def _cpu_model():
    """The host CPU's model name (lscpu), else what /proc/cpuinfo names."""
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


# ---- our arm ------------------------------------------------------------------------------------

# the files the tensor-core decode kernel and its launch are compiled from: the recorded
# ncu traffic stays valid until one of them changes
DECODE_KERNEL_SOURCES = ("decode_mma.cu", "decode_flat.cu", "paged_decode_mma.cuh",
                         "decode_epilogue.cuh", "decode_plan.cuh", "combine_merge.cuh",
                         "pkv_device.cuh", "pkv_internal.h", "capi.cu")


def source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_271_gb300", "csrc")
    for fn in DECODE_KERNEL_SOURCES:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(split):
    """dram bytes per launch of the decode kernel from the committed ncu summary, if it was
    taken on the current kernel sources and on the split this run used; else None."""
    path = os.path.join(ROOT, "profiles", "paged_decode_llama3_8b_b64.traffic.txt")
    try:
        with open(path) as f:
            rec = dict(tok.split("=", 1) for tok in f.read().split())
        if rec.get("source_sha") == source_sha() and split.split(" ")[0] == rec.get("split"):
            return float(rec["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def set_split(pkv, args):
    """auto: the decode's split (chunks, longer chunks or balanced) is measured on the first
    call of the shape (autotuning); otherwise the one named."""
    if args.split == "auto":
        pkv.decode_set_autotune(True)
    else:
        pkv.decode_set_split({"chunks": 1, "balanced": 2, "chunks-x1.5": 3, "chunks-x2": 4}[args.split])


def run_ours(args):
    import torch
    import paged_kv_cache_271_gb300 as pkv

    ws, rank, local = rank_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    pkv.lib()  # fail loudly if the library is missing
    set_split(pkv, args)

    sc = StepState(args.workload, dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(FLUSH_BYTES if args.l2 == "flush" else 0, dev)
    n_sets = 1
    sc.config["l2"] = "flushed with a 256 MiB write before every timed step"
    if args.l2 == "rotate":
        # Inputs larger than the L2 instead of a flush (whose dirty lines would be written back
        # inside the timed step): identical copies of the pools, used in turn, so that a copy
        # is read again only after at least 3 x L2 bytes of other copies.
        used = sc.used_kv_bytes()
        n_sets = max(2, int(math.ceil(3 * L2_BYTES / used)))
        sc.make_copies(n_sets)
        sc.config["l2"] = ("not flushed: %d copies of the KV pools (%.0f MB of pages in use "
                           "each) used in turn, %.0f MB of other copies read between two reads "
                           "of one copy (L2: 129 MB)" % (n_sets, used / 1e6,
                                                           (n_sets - 1) * used / 1e6))
    per_step_bytes = sc.decode_bytes() + sc.append_bytes()
    step_host = sc.host_step

    for i in range(args.warmup):
        flush.zero_()
        step_host()
        sc.fused_step(pool=i % n_sets)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    sc.config["split"] = (sc.split_label() if args.split == "auto"
                          else args.split + " (fixed by --split)")

    # The step's device work (append, decode, combine) is captured once as a CUDA graph (one
    # per pool copy) and replayed every step, as a serving loop would; the host slot mapping
    # runs outside it.
    graphs = []
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(3):
            sc.fused_step(pool=i % n_sets)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    for p in range(n_sets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sc.fused_step(pool=p)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        flush.zero_()
        graphs[i % n_sets].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    host_s = 0.0
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        t0 = time.perf_counter()
        step_host()
        host_s += time.perf_counter() - t0
        starts[i].record(stream)
        graphs[i % n_sets].replay()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_step = float(np.mean(ms))
    assert pkv.device_error() == 0

    # The other L2 treatment, for comparison: a 256 MiB write before every step (rotate mode),
    # or no flush and one pool copy (flush mode).
    alt = L2Flush(FLUSH_BYTES if args.l2 == "rotate" else 0, dev)
    a_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    a_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        alt.zero_()
        a_starts[i].record(stream)
        graphs[0].replay()
        a_ends[i].record(stream)
    torch.cuda.synchronize()
    alt_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(a_starts, a_ends)]))
    del alt

    # Per-kernel durations: the same steps launched directly with the library's tracing on
    # (events on the launching stream around every kernel).
    pkv.trace_reset()
    pkv.trace_enable(True)
    for i in range(args.steps):
        flush.zero_()
        sc.fused_step(pool=i % n_sets)
    torch.cuda.synchronize()
    pkv.trace_enable(False)
    launches = {}
    for k in ("kv_append", "cascade_prefix", "paged_decode", "decode_combine"):
        launches[k] = pkv.trace_read(k)
    pkv.trace_reset()
    per_step_launches = sum(n for n, _ in launches.values()) / max(args.steps, 1)
    assert pkv.device_error() == 0

    max_ms = max_over_ranks(ms_step, dev)
    value = aggregate(per_step_bytes, max_ms, ws)
    hbm_peak, peak_kind = peaks()

    # the roofline of the kernel that takes the most time in the step
    work = sc.kernel_work()
    top = max(work, key=lambda k: launches[k][1])
    n_top, t_top = launches[top]
    top_ms = t_top / max(n_top, 1)
    if work[top][0] == "hbm":
        kernel_bytes = work[top][1]
        achieved = kernel_bytes / (top_ms * 1e-3) / 1e9
        traffic = (recorded_traffic(sc.config.get("split", ""))
                   if args.workload == "llama3_8b_b64" else None)
        roofline = {"bound": "hbm",
                    "kernel": "paged_decode kernel (%s cache, d=%d, G=%d, append fused; "
                              "split: %s)" % (sc.config["kv_dtype"], sc.d, sc.h_q // sc.h_kv,
                                              sc.config.get("split", "chunks")),
                    "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                    "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                    "traffic": traffic, "algorithmic_bytes_per_launch": kernel_bytes,
                    "launch_ms": round(top_ms, 5)}
    else:
        flops, byts = work[top][1], work[top][2]
        tf_peak, tf_kind = peaks("bf16_tflops")
        achieved = flops / (top_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "cascade_prefix kernel (bf16 tcgen05, d=%d)" % sc.d,
                    "achieved": round(achieved, 2), "peak": tf_peak, "unit": "TFLOP/s",
                    "frac": round(achieved / tf_peak, 4), "peak_kind": tf_kind + " cuBLAS bf16",
                    "traffic": None, "algorithmic_flops_per_launch": flops,
                    "algorithmic_bytes_per_launch": byts,
                    "bytes_GBs": round(byts / (top_ms * 1e-3) / 1e9, 1),
                    "launch_ms": round(top_ms, 5)}
    roofline["other_kernels"] = {
        k: {"bound": v[0], "ms": round(launches[k][1] / max(launches[k][0], 1), 5),
            ("GB/s" if v[0] == "hbm" else "TFLOP/s"): round(
                v[1] / (launches[k][1] / max(launches[k][0], 1) * 1e-3) / (1e9 if v[0] == "hbm" else 1e12), 2)}
        for k, v in work.items() if k != top and launches[k][0]}

    roofline["sm_mhz"] = clk.get("sm_mhz")  # median SM clock sampled during the timed steps
    e2e = run_e2e(sc, args, dev, stream, flush, n_sets)
    max_e2e = max_over_ranks(e2e["ms_per_step"], dev)
    e2e_value = aggregate(per_step_bytes, max_e2e, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.workload == "llama3_8b_b64":
        cpu = cpu_baseline(workload())

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if sc.kv_bytes == 2 else (sc.config["kv_dtype"] + "/f16" if sc.kv_bytes == 1 else "f32"),
            "data": "synthetic", "config": dict(sc.config, parallelism="replicas x%d" % ws),
            "decode_tokens_per_s": round(ws * sc.batch / (max_ms * 1e-3), 1),
            "tokens_per_s_32_layer_projection": round(ws * sc.batch / (32 * max_ms * 1e-3), 1),
            "steps_per_s": round(1e3 / max_ms, 1),
            "unique_bytes_GBs": round(ws * sc.unique_bytes() / (max_ms * 1e-3) / 1e9, 1),
            ("l2_flushed" if args.l2 == "rotate" else "l2_not_flushed"): {
                "ms_per_step": round(alt_ms, 5),
                "value": round(aggregate(per_step_bytes, alt_ms, 1) * ws, 1)},
            "pct_of_peak": {"measured_copy_%s" % peak_kind: round(100 * value / ws / hbm_peak, 2),
                            "nominal_8TBs": round(100 * value / ws / NOMINAL_HBM_GBS, 2)},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "ms_per_step": round(max_e2e, 5),
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "phases_us": e2e["phases_us"]},
            "gpu_launches": int(round(per_step_launches * args.steps)),
            "graph": "the step's launches captured once as a CUDA graph, replayed per step",
            "host_slot_mapping_us": round(1e6 * host_s / max(args.steps, 1), 1),
            "host_step": "slot mapping" + (" + cascade grouping" if sc.groups is not None else ""),
            "launches_per_kernel": {k: n for k, (n, _) in launches.items()},
            "kernel_ms": {k: round(t / max(n, 1), 5) for k, (n, t) in launches.items()},
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)


class L2Flush:
    """zero_() writes a buffer larger than the L2 (nothing when size is 0)."""

    def __init__(self, size, dev):
        import torch
        self.buf = torch.empty(size, dtype=torch.uint8, device=dev) if size else None

    def zero_(self):
        if self.buf is not None:
            self.buf.zero_()


def run_prompt_append(args):
    """The prompt prefill of replacement requests in the continuous-batching workload through
    the quantising append alone: 20 prompts of U[128, 2048] tokens (seeded), bf16 K/V rows
    already on the device (three input sets used in turn, 250 MB: more than the L2), quantised
    with per-head scales into an FP8 (or INT8) pool at slots the request tables hand out. A
    step is one kv_append launch; ``value`` is its bytes (bf16 rows read, codes written) over
    the step time. ``e2e`` adds the copy of the rows and slots from pinned host memory."""
    import torch
    import paged_kv_cache_271_gb300 as pkv
    from paged_kv_cache_271_gb300.cache import PagedKVCache
    ws, rank, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    pkv.lib()
    i8 = args.workload.startswith("int8")
    h_kv, d = 8, 128
    rng = np.random.default_rng(271005)
    lens = rng.integers(128, 2049, 20)
    n = int(lens.sum())
    pages = int(sum(pkv.pages_needed(int(x)) for x in lens) * 1.1) + 1
    g = torch.Generator().manual_seed(271005)
    sets = [(torch.randn(n, h_kv, d, generator=g).to(torch.bfloat16).to(dev),
             torch.randn(n, h_kv, d, generator=g).to(torch.bfloat16).to(dev)) for _ in range(3)]
    ks = pkv.kv_absmax_scales(sets[0][0], int8=i8)
    vs = pkv.kv_absmax_scales(sets[0][1], int8=i8)
    cache = PagedKVCache(pages, h_kv, d, torch.int8 if i8 else torch.float8_e4m3fn, dev,
                         initial_free_order=rng.permutation(pages), k_scales=ks, v_scales=vs)
    rids = list(range(len(lens)))
    for r in rids:
        cache.add_request(r)
    slots_host = cache.reserve(rids, [int(x) for x in lens])
    slots = torch.from_numpy(slots_host).to(dev)
    byts = 2 * n * h_kv * d * (2 + 1)

    def step(i, stream=None):
        k, v = sets[i % 3]
        pkv.kv_append(k, v, slots, cache.k, cache.v, ks, vs, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        st[i].record(stream)
        step(i)
        en[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)]))
    assert pkv.device_error() == 0
    max_ms = max_over_ranks(ms, dev)
    hbm_peak, peak_kind = peaks()
    value = aggregate(byts, max_ms, ws)

    # e2e: the step's rows and slots copied from pinned host memory, then the append
    hk = [torch.empty((n, h_kv, d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hk[0].copy_(sets[0][0].cpu())
    hk[1].copy_(sets[0][1].cpu())
    hs = torch.from_numpy(slots_host).pin_memory()
    dk, dv, dsl = torch.empty_like(sets[0][0]), torch.empty_like(sets[0][1]), torch.empty_like(slots)
    for i in range(3):
        dk.copy_(hk[0], non_blocking=True)
        dv.copy_(hk[1], non_blocking=True)
        dsl.copy_(hs, non_blocking=True)
        pkv.kv_append(dk, dv, dsl, cache.k, cache.v, ks, vs)
    torch.cuda.synchronize()
    e_st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        e_st[i].record(stream)
        dk.copy_(hk[0], non_blocking=True)
        dv.copy_(hk[1], non_blocking=True)
        dsl.copy_(hs, non_blocking=True)
        pkv.kv_append(dk, dv, dsl, cache.k, cache.v, ks, vs)
        e_en[i].record(stream)
        e_en[i].synchronize()
    barrier()
    e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(e_st, e_en)])), dev)
    assert pkv.device_error() == 0
    if rank == 0:
        coded = "int8" if i8 else "fp8_e4m3"
        print(json.dumps({
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16->" + coded, "data": "synthetic",
            "config": {"workload": "%s_prompt_append_20_prompts" % coded.split("_")[0],
                       "prompt_lens": "U[128, 2048] seeded, sum %d" % n, "num_kv_heads": h_kv,
                       "head_dim": d, "page_size": 16, "kv_dtype": coded, "pool_pages": pages,
                       "l2": "not flushed: 3 input sets of %.0f MB used in turn" % (
                           2 * n * h_kv * d * 2 / 1e6),
                       "step": "device: one quantising kv_append launch (bf16 rows in, codes "
                               "written at the requests' slots)",
                       "parallelism": "replicas x%d" % ws},
            "roofline": {"bound": "hbm", "kernel": "kv_append (bf16 -> %s)" % coded,
                         "achieved": round(value / ws, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(value / ws / hbm_peak, 4), "peak_kind": peak_kind,
                         "traffic": None, "algorithmic_bytes_per_launch": byts,
                         "launch_ms": round(max_ms, 5), "sm_mhz": clk.get("sm_mhz")},
            "cpu_baseline": None,
            "e2e": {"value": round(aggregate(byts, e2e_ms, ws), 1), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": 2 * n * h_kv * d * 2 + 8 * n,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": args.steps, "clocks": clk}), flush=True)


def run_fork(args):
    """Copy-on-write fork (parallel sampling): per step, fork each of 16 prompts into 4 samples
    (reference counts), reserve each sample's first slot -- the shared, partly filled last page
    of its prompt is copied for every writer (pkv_cow_page on the host, pkv_copy_pages on the
    device) --, run the fused append + decode over the 64 samples, and free the samples again,
    so that every step starts from the same state. ``value`` counts the decode's bytes plus the
    copied pages (read and written)."""
    import torch
    import paged_kv_cache_271_gb300 as pkv
    from paged_kv_cache_271_gb300.cache import PagedKVCache
    import workloads
    ws, rank, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    pkv.lib()
    ps = workloads.parallel_sampling()
    w = ps.prompts
    cache = PagedKVCache(w.num_pages, w.num_kv_heads, w.head_dim, torch.bfloat16, dev,
                         initial_free_order=w.page_order)
    P, S = w.batch, ps.samples
    for p in range(P):
        cache.add_request(p)
    slots = cache.reserve(list(range(P)), [int(n) for n in w.context_lens])
    cache.write(slots, w.k_tokens.to(dev), w.v_tokens.to(dev))
    q, k_new, v_new = ps.q.to(dev), ps.k_new.to(dev), ps.v_new.to(dev)
    rids = [1000 + i for i in range(P * S)]
    out = torch.empty_like(q)
    maxp = int(max(pkv.pages_needed(int(n) + 1) for n in w.context_lens))
    need = pkv.decode_workspace_size(P * S, 32, 8, 128, maxp)
    workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    bt_dev = torch.zeros((P * S, maxp), dtype=torch.int32, device=dev)
    cl_dev = torch.zeros((P * S,), dtype=torch.int32, device=dev)
    bt_pin = torch.zeros((P * S, maxp), dtype=torch.int32).pin_memory()
    cl_pin = torch.zeros((P * S,), dtype=torch.int32).pin_memory()
    out_pin = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    copies = [0]
    cp_pin = torch.zeros((2, P * S), dtype=torch.int32).pin_memory()
    cp_dev = torch.zeros((2, P * S), dtype=torch.int32, device=dev)

    parents = np.arange(P * S, dtype=np.int64) // S
    rids = np.asarray(rids, dtype=np.int64)
    ones = np.ones(P * S, dtype=np.int32)
    cp_np = cp_pin.numpy()

    def host_fork():
        cache.fork_many(parents, rids)
        pairs = []
        cache.reserve(rids, ones, copies_out=pairs)  # copy-on-write decisions
        copies[0] = len(pairs)
        if pairs:
            cp_np[:, :len(pairs)] = np.asarray(pairs, dtype=np.int32).T
        cache.block_table_array(rids, maxp, out=bt_pin)  # straight into the pinned buffers
        cache.context_lens_array(rids, out=cl_pin)

    def device_step():
        cp_dev.copy_(cp_pin, non_blocking=True)
        bt_dev.copy_(bt_pin, non_blocking=True)
        cl_dev.copy_(cl_pin, non_blocking=True)
        n = copies[0]
        if n:
            pkv.copy_pages(cache.k, cache.v, cp_dev[0, :n], cp_dev[1, :n])
        pkv.paged_decode_step(q, k_new, v_new, cache.k, cache.v, bt_dev, cl_dev, w.scale,
                              out=out, workspace=workspace)

    def host_free():
        cache.free_many(rids)

    for _ in range(args.warmup):
        host_fork()
        device_step()
        torch.cuda.synchronize()
        host_free()
    assert pkv.device_error() == 0
    # The device step (the three table copies from pinned buffers, the page copies, the fused
    # append + decode, the combine) is captured once as a CUDA graph and replayed every step, as
    # for the other workloads. The fork pattern is the same every step, so is the number of
    # copied pages; the graph is re-captured if it ever changes.
    graph = [None, -1]

    def replay():
        if copies[0] != graph[1]:
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                device_step()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                device_step()
            torch.cuda.synchronize()
            graph[0], graph[1] = g, copies[0]
        graph[0].replay()

    for _ in range(max(3, args.warmup)):
        host_fork()
        replay()
        torch.cuda.synchronize()
        host_free()
    assert pkv.device_error() == 0
    n = args.steps
    dev_ms, host_s, e2e_ms = [], 0.0, []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    for i in range(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        host_fork()  # host: fork, copy-on-write decisions, tables (timed on the host)
        th = time.perf_counter() - t0
        host_s += th
        e0.record(stream)
        replay()
        e1.record(stream)
        out_pin.copy_(out, non_blocking=True)
        e2.record(stream)
        e2.synchronize()
        dev_ms.append(e0.elapsed_time(e1))
        e2e_ms.append(1e3 * th + e0.elapsed_time(e2))  # host bookkeeping + copies + step + D2H
        host_free()
    barrier()
    clk = clocks.stop()
    assert pkv.device_error() == 0
    ctx = [int(cache.lens[p]) + 1 for p in range(P) for _ in range(S)]
    row = 8 * 128 * 2 * 2
    decode_bytes = sum(ctx) * row + 2 * P * S * 32 * 128 * 2 + 2 * P * S * 8 * 128 * 4
    copy_bytes = copies[0] * 8 * 16 * 128 * 2 * 2 * 2  # pages x (K and V) x (read and write)
    ms = max_over_ranks(float(np.mean(dev_ms)), dev)
    e2e = max_over_ranks(float(np.mean(e2e_ms)), dev)
    peak, kind = peaks()
    if rank == 0:
        value = aggregate(decode_bytes + copy_bytes, ms, ws)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "prompts": P, "samples_per_prompt": S,
                       "batch": P * S, "num_q_heads": 32, "num_kv_heads": 8, "head_dim": 128,
                       "page_size": 16, "kv_dtype": "bf16",
                       "prompt_lens": "U[1000, 3000], sum %d" % int(np.sum(w.context_lens)),
                       "step": "device: table copies + copy-on-write page copies + fused append "
                               "+ decode (host fork, copy-on-write decisions and tables timed "
                               "apart, host_fork_us); samples freed after each step",
                       "l2": "not flushed: the step reads the prompts' pages (%.0f MB) once"
                             % (sum(int(x) for x in w.context_lens) * row / 1e6),
                       "parallelism": "replicas x%d" % ws},
            "copied_pages_per_step": copies[0],
            "decode_tokens_per_s": round(ws * P * S / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "kernel": "page copies + paged_decode step (device)",
                         "achieved": round(value / ws, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(value / ws / peak, 4), "peak_kind": kind, "traffic": None,
                         "algorithmic_bytes_per_launch": decode_bytes + copy_bytes,
                         "launch_ms": round(ms, 5)},
            "cpu_baseline": None,
            "host_fork_us": round(1e6 * host_s / n, 1),
            "host_fork": "native request tables (pkv_seq_*): 64 forks, copy-on-write reserve, "
                         "tables into pinned buffers",
            "e2e": {"value": round(aggregate(decode_bytes + copy_bytes, e2e, ws), 1), "unit": "GB/s",
                    "ms_per_step": round(e2e, 5),
                    "h2d_bytes_per_step": int(bt_pin.numel() * 4 + cl_pin.numel() * 4),
                    "d2h_bytes_per_step": int(out.numel() * 2)},
            "gpu_launches": int(3 * n), "clocks": clk,
            "graph": "the device step captured once as a CUDA graph, replayed per step",
        }
        print(json.dumps(line), flush=True)


def run_e2e(sc, args, dev, stream, flush, n_sets=1):
    """Same step through the public API from pinned host buffers (pkv.HostStep): per step one
    host->device copy of the step's inputs (queries, new K/V rows, page tables, context
    lengths; for the cascade also this step's groups, which the library finds on the host from
    the tables inside the same call) and the device->host copy of the outputs sit inside the
    timed region, and the host waits for the outputs before the next step."""
    import torch
    import paged_kv_cache_271_gb300 as pkv
    cascade = sc.groups is not None
    hs = pkv.HostStep(sc.batch, sc.h_q, sc.h_kv, sc.d, sc.bt.shape[1], q_dtype=sc.q.dtype,
                      new_dtype=sc.k_new.dtype, device=dev, cascade=cascade)
    hs.q_host.copy_(sc.q.cpu())
    hs.k_new_host.copy_(sc.k_new.cpu())
    hs.v_new_host.copy_(sc.v_new.cpu())
    hs.block_tables_host.copy_(sc.bt.cpu())
    hs.context_lens_host.copy_(sc.cl.cpu())
    ks, vs = sc.scales if sc.scales else (None, None)

    def one(i):
        k, v = sc.pools[i % n_sets] if hasattr(sc, "pools") else (sc.k, sc.v)
        if cascade:  # this step's groups found by the library from the packed host tables
            hs.cascade_step(k, v, sc.scale, sc.workspace)
        else:
            hs.step(k, v, sc.scale, k_scales=ks, v_scales=vs, workspace=sc.workspace,
                    window=getattr(sc, "window", 0), sink_tokens=getattr(sc, "sink", 0))

    for i in range(max(3, args.warmup)):
        flush.zero_()
        one(i)
    torch.cuda.synchronize()
    n = max(1, args.steps)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    barrier()
    torch.cuda.synchronize()
    for i in range(n):
        flush.zero_()
        starts[i].record(stream)
        one(i)
        ends[i].record(stream)
        ends[i].synchronize()  # the result is on the host before the next step starts
    barrier()
    ms = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))

    # Where an e2e step's time goes, from the same steps run again: host time inside the
    # library call (argument marshalling, grouping for the cascade, enqueueing the copies and
    # launches) and waiting for the output; device time of each copy and kernel (the library's
    # event tracing); the rest of the step's device-side span is time the GPU sat idle
    # between them (waiting for the host to enqueue, copy and launch latencies).
    t_call = t_wait = 0.0
    pkv.trace_reset()
    pkv.trace_enable(True)
    for i in range(n):
        flush.zero_()
        t0 = time.perf_counter()
        one(i)
        t1 = time.perf_counter()
        torch.cuda.current_stream().synchronize()
        t_call += t1 - t0
        t_wait += time.perf_counter() - t1
    pkv.trace_enable(False)
    phases = {"host_call": round(1e6 * t_call / n, 2), "host_wait": round(1e6 * t_wait / n, 2)}
    busy = 0.0
    for k in ("h2d_copy", "cascade_prefix", "paged_decode", "decode_combine", "d2h_copy"):
        cnt, tot = pkv.trace_read(k)
        if cnt:
            phases[k] = round(1e3 * tot / n, 2)
            busy += 1e3 * tot / n
    pkv.trace_reset()
    phases["gpu_idle"] = round(1e3 * ms - busy, 2)
    return {"ms_per_step": ms, "h2d": hs.h2d_bytes, "d2h": hs.d2h_bytes, "phases_us": phases}


def trace_joins(tr):
    """Per step of a continuous-batching trace, the requests that join before it: (slot,
    finished request, new request) triples, from the trace's finish flags and request table."""
    return [[] if s == 0 else
            [(b, int(tr.rid_table[s - 1, b]), int(tr.rid_table[s, b]))
             for b in range(tr.batch) if tr.finish[s - 1, b]] for s in range(tr.steps)]


def trace_bookkeeping(cache, tr, joins, rid_arr, width, tables_out, lens_out):
    """One step's scheduler bookkeeping for a continuous-batching trace, in one library call
    (PagedKVCache.step -> pkv_seq_step): the finished requests of ``joins`` (slot, finished,
    new) are freed, the new ones take their slots in ``rid_arr`` and get room for their
    prompts, every live request gets room for one token, and the live requests' table rows
    (patched in place where a slot keeps its request) and lengths go to ``tables_out`` /
    ``lens_out``. Returns the prompts' slots, request by request in ``joins`` order."""
    old = np.array([o for _, o, _ in joins], dtype=np.int64)
    new = np.array([r for _, _, r in joins], dtype=np.int64)
    for b, _, rid in joins:
        rid_arr[b] = rid
    slots, _, _ = cache.step(old, new, tr.prompt_lens[new], rid_arr, width,
                             tables_out=tables_out, lens_out=lens_out, incremental=True)
    return slots


def run_trace(args):
    """FP8 (or INT8) continuous batching over the whole trace: 256 request slots, contexts
    U[128, 8192] at the start; every step each live request gains one token, and a request
    that finished (probability 0.05 per step) is freed and replaced by a new one whose prompt
    (U[128, 2048] tokens) is prefilled through the quantising append. ``--warmup`` steps run
    first, untimed; the trace is ``warmup + steps`` long.

    A step is: the host bookkeeping (frees, new requests, the prompts' and the new tokens'
    slots, page tables and context lengths into pinned buffers: native request tables, timed
    on the host); the copies of the step's inputs from pinned host memory (queries, new K/V
    rows, the prompts' K/V rows, tables, context lengths, prompt slots); the device work (the
    prompts' quantising append, the fused append + decode of every live request, the combine);
    the copy of the output to the host. ``value`` is the step's algorithmic bytes (K and V of
    every attended token, queries, outputs, appended rows, prompt rows) over the device work
    alone (its inputs resident by then); ``e2e`` over host bookkeeping + copies + device work."""
    import torch
    import paged_kv_cache_271_gb300 as pkv
    import workloads
    from gpu_harness import ContinuousBatchingRun
    ws, rank, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    pkv.lib()
    set_split(pkv, args)
    coded = "int8" if args.workload.startswith("int8") else "fp8_e4m3"
    n_warm, n = max(3, args.warmup), max(1, args.steps)
    tr = workloads.fp8_continuous_batching(steps=n_warm + n)
    run = ContinuousBatchingRun(tr, device=dev, cache_dtype=coded)  # scales + initial prefill
    cache, B, h_q, h_kv, d = run.cache, tr.batch, tr.num_q_heads, tr.num_kv_heads, tr.head_dim
    joins_at = trace_joins(tr)
    n_max = max(1, max(sum(int(tr.prompt_lens[r]) for _, _, r in j) for j in joins_at))
    width = pkv.pages_needed(int(tr.prompt_lens.max()) + tr.steps)
    need = pkv.decode_workspace_size(B, h_q, h_kv, d, width)
    workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    bf = torch.bfloat16

    def pair(shape, dtype):
        return (torch.zeros(shape, dtype=dtype).pin_memory(),
                torch.zeros(shape, dtype=dtype, device=dev))

    bt = pair((B, width), torch.int32)
    cl = pair((B,), torch.int32)
    ps = pair((n_max,), torch.int64)
    q = pair((B, h_q, d), bf)
    kn, vn = pair((B, h_kv, d), bf), pair((B, h_kv, d), bf)
    kp, vp = pair((n_max, h_kv, d), bf), pair((n_max, h_kv, d), bf)
    out = torch.empty((B, h_q, d), dtype=bf, device=dev)
    out_pin = torch.empty(out.shape, dtype=bf).pin_memory()
    stream = torch.cuda.current_stream()
    start_step = {b: 0 for b in range(B)}  # request -> the step it joined
    expect = np.zeros(B, dtype=np.int32)
    rid_arr = np.arange(B, dtype=np.int64)  # the live request of each slot

    def stage(s):
        """Step s's inputs into the pinned buffers (untimed): queries, every live request's
        new K/V row and the prompts of the requests that join before it."""
        o = 0
        for _, old, rid in joins_at[s]:
            del run.tokens[old]
            run.tokens[rid] = tr.request_tokens(rid)
            start_step[rid] = s
            m = int(tr.prompt_lens[rid])
            kp[0][o:o + m].copy_(run.tokens[rid][0][:m])
            vp[0][o:o + m].copy_(run.tokens[rid][1][:m])
            o += m
        rids = [int(r) for r in tr.rid_table[s]]
        pos = [int(tr.prompt_lens[r]) + s - start_step[r] for r in rids]
        expect[:] = np.asarray(pos, dtype=np.int32) + 1  # the lengths the tables must give
        kn[0].copy_(torch.stack([run.tokens[r][0][p] for r, p in zip(rids, pos)]))
        vn[0].copy_(torch.stack([run.tokens[r][1][p] for r, p in zip(rids, pos)]))
        q[0].copy_(tr.step_q(s))

    def host(s):
        """Frees, new requests, slots, tables: the bookkeeping a scheduler does per step."""
        for b, _, rid in joins_at[s]:  # a new request takes the finished one's slot
            run.slot_rid[b] = rid
        slots = trace_bookkeeping(cache, tr, joins_at[s], rid_arr, width, bt[0], cl[0])
        npr = len(slots)
        if npr:
            ps[0].numpy()[:npr] = slots
        return npr

    def copy_in(npr):
        for h, dv in (q, kn, vn, bt, cl):
            dv.copy_(h, non_blocking=True)
        if npr:
            for h, dv in (kp, vp, ps):
                dv[:npr].copy_(h[:npr], non_blocking=True)

    def device(npr):
        if npr:
            pkv.kv_append(kp[1][:npr], vp[1][:npr], ps[1][:npr], cache.k, cache.v,
                          run.k_scales, run.v_scales)
        pkv.paged_decode_step(q[1], kn[1], vn[1], cache.k, cache.v, bt[1], cl[1], tr.scale,
                              out=out, k_scales=run.k_scales, v_scales=run.v_scales,
                              workspace=workspace)
        return 2 + (1 if npr else 0)  # the fused step, the combine, the prompts' append

    for s in range(n_warm):
        stage(s)
        npr = host(s)
        assert np.array_equal(cl[0].numpy(), expect), s
        copy_in(npr)
        device(npr)
        torch.cuda.synchronize()
    assert pkv.device_error() == 0
    row = h_kv * d * 1 * 2  # K and V codes of one token
    app = 2 * h_kv * d * (2 + 1)  # a bf16 row in and a code row out, K and V
    dev_ms, e2e_ms, host_s, byts, h2d, launches, n_prompt_tok, n_joins = [], [], 0.0, 0, 0, 0, 0, 0
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    for s in range(n_warm, n_warm + n):
        stage(s)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        t0 = time.perf_counter()
        npr = host(s)
        th = time.perf_counter() - t0
        ev[0].record(stream)
        copy_in(npr)
        ev[1].record(stream)
        launches += device(npr)
        ev[2].record(stream)
        out_pin.copy_(out, non_blocking=True)
        ev[3].record(stream)
        ev[3].synchronize()
        host_s += th
        assert np.array_equal(cl[0].numpy(), expect), s  # tables agree with the trace
        dev_ms.append(ev[1].elapsed_time(ev[2]))
        e2e_ms.append(1e3 * th + ev[0].elapsed_time(ev[3]))
        byts += int(cl[0].sum()) * row + 2 * B * h_q * d * 2 + B * app + npr * app
        h2d += (q[0].numel() + kn[0].numel() + vn[0].numel()) * 2 + (bt[0].numel() + B) * 4 \
            + npr * (2 * h_kv * d * 2 + 8)
        n_prompt_tok += npr
        n_joins += len(joins_at[s])
    barrier()
    clk = clocks.stop()
    # Per-kernel durations: the last step's device work again (it rewrites the same slots with
    # the same values), with the library's tracing on and the L2 flushed before each repeat.
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pkv.trace_reset()
    pkv.trace_enable(True)
    for _ in range(10):
        flush.zero_()
        device(npr)
    torch.cuda.synchronize()
    pkv.trace_enable(False)
    kernel_ms = {}
    for k in ("kv_append", "paged_decode", "decode_combine"):
        c, t = pkv.trace_read(k)
        kernel_ms[k] = round(t / max(c, 1), 5)
    pkv.trace_reset()
    del flush
    assert pkv.device_error() == 0
    ms = max_over_ranks(float(np.mean(dev_ms)), dev)
    e2e = max_over_ranks(float(np.mean(e2e_ms)), dev)
    per_step = byts / n
    peak, kind = peaks()
    if rank == 0:
        value = aggregate(per_step, ms, ws)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": n, "warmup": n_warm, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": coded + "/bf16", "data": "synthetic",
            "config": {"workload": ("int8" if coded == "int8" else "fp8")
                       + "_continuous_batching_b%d_trace" % B, "batch": B, "num_q_heads": h_q,
                       "num_kv_heads": h_kv, "head_dim": d, "page_size": 16, "kv_dtype": coded,
                       "trace_steps": tr.steps,
                       "timed_steps": "%d..%d" % (n_warm, n_warm + n - 1),
                       "context_lens": "initial U[128, 8192]; replacements U[128, 2048]; "
                                       "finish p = 0.05 per step",
                       "pool_pages": tr.num_pages,
                       "step": "device: quantising prompt append + fused append + decode + "
                               "combine (host bookkeeping and the copies in e2e only)",
                       "l2": "not flushed: a step reads %.0f MB of pages (L2: 129 MB)"
                             % (per_step / 1e6),
                       "parallelism": "replicas x%d" % ws},
            "steps_per_s": round(1e3 / ms, 1),
            "decode_tokens_per_s": round(ws * B / (ms * 1e-3), 1),
            "prompt_tokens_per_step": round(n_prompt_tok / n, 1),
            "requests_replaced": n_joins,
            "roofline": {"bound": "hbm", "kernel": "whole device step (append + decode + combine)",
                         "achieved": round(value / ws, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(value / ws / peak, 4), "peak_kind": kind, "traffic": None,
                         "algorithmic_bytes_per_launch": int(per_step), "launch_ms": round(ms, 5)},
            "cpu_baseline": None,
            "host_step_us": round(1e6 * host_s / n, 1),
            "kernel_ms": kernel_ms,
            "kernel_ms_of": "the last timed step's device work run 10 more times, one event "
                            "pair per kernel, L2 flushed before each (%d prompt tokens)" % npr,
            "e2e": {"value": round(aggregate(per_step, e2e, ws), 1), "unit": "GB/s",
                    "ms_per_step": round(e2e, 5), "h2d_bytes_per_step": int(h2d / n),
                    "d2h_bytes_per_step": int(out.numel() * 2)},
            "gpu_launches": int(launches), "clocks": clk,
            "graph": "none: the step's shapes change along the trace (launched op by op)",
        }
        print(json.dumps(line), flush=True)


# ---- reference arm: the oracle as it stands --------------------------------------------------

def run_reference(args):
    ws, rank, _ = rank_info()
    if rank != 0:
        return
    import oracle
    w = workload("llama3_8b_b64")
    threads = oracle.max_threads()
    n_seq = 2
    for _ in range(args.warmup):
        oracle_sample(w, n_seq)
    times, byts = [], 0
    for _ in range(args.steps):
        byts, t = oracle_sample(w, n_seq)
        times.append(t)
    ms = float(np.mean(times)) * 1e3
    value = byts / (ms * 1e-3) / 1e9
    sample = ("fp64 C oracle paged decode of the first %d of %d requests (all heads) per step"
              % (n_seq, w.batch))
    line = {"metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": dict(config_of(w), parallelism="host cores",
                           l2="not applicable: the oracle runs on the host cores",
                           step="fp64 oracle paged decode over each sampled request's cached and "
                                "new tokens (the append is its host scatter, untimed)"),
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample, "cpu": _cpu_model()},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                    help="rotate: copies of the pools used in turn (at least 3 x L2 of other "
                         "copies between two reads of one); flush: write 256 MiB before every "
                         "timed step")
    ap.add_argument("--split", choices=["auto", "chunks", "balanced", "chunks-x1.5", "chunks-x2"],
                    default="auto", help="the decode's split: measured per shape (auto) or fixed")
    ap.add_argument("--workload", choices=WORKLOADS, default="llama3_8b_b64",
                    help="the default is the headline layer; the others are for measurement")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("bench.py: at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "parallel_sampling_fork":
        run_fork(args)
    elif args.workload in ("fp8_cb_trace", "int8_cb_trace"):
        run_trace(args)
    elif args.workload in ("fp8_prompt_append", "int8_prompt_append"):
        run_prompt_append(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
