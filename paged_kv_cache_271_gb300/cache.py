"""One layer's paged KV cache: the two pools plus the host bookkeeping around them.

"KV cache and PagedAttention", section 4: a physical pool of fixed-size pages and, per
request, a page table listing its pages; the allocator is O(1); requests with a common
prefix point at the same pages (reference-counted here). Section 5 (continuous batching):
requests join and leave the running batch every step, so pages are freed and reused.

Page accounting, slot mapping and the allocator run in the C library (``pkv_pages_needed``,
``pkv_slot_mapping``, ``pkv_alloc``/``pkv_incref``/``pkv_decref``); this class only keeps the
per-request page lists and hands tensors to the kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import PageAllocator, PkvError, copy_pages, kv_append, pages_needed, slot_mapping


class PagedKVCache:
    def __init__(self, num_pages: int, num_kv_heads: int, head_dim: int, dtype: torch.dtype,
                 device="cuda", page_size: int = 16, initial_free_order=None,
                 k_scales: torch.Tensor | None = None, v_scales: torch.Tensor | None = None):
        if dtype == torch.float8_e4m3fn:
            dtype = torch.uint8  # FP8 E4M3 codes; torch.int8 pools hold INT8 codes
        self.k = torch.empty(num_pages, num_kv_heads, page_size, head_dim, dtype=dtype,
                             device=device)
        self.v = torch.empty_like(self.k)
        self.page_size = page_size
        self.num_pages = num_pages
        self.allocator = PageAllocator(num_pages, initial_free_order)
        self.k_scales = k_scales
        self.v_scales = v_scales
        self.pages: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    @property
    def is_fp8(self) -> bool:
        return self.k.dtype == torch.uint8

    @property
    def is_int8(self) -> bool:
        return self.k.dtype == torch.int8

    # ---- requests ---------------------------------------------------------------------------

    def add_request(self, rid: int, shared_pages=None, shared_len: int = 0):
        """New request; optionally starting on ``shared_pages`` that already hold its first
        ``shared_len`` tokens (a prefix, whole pages only)."""
        if rid in self.pages:
            raise PkvError(-1, "request %d exists" % rid)
        pages = [] if shared_pages is None else [int(p) for p in shared_pages]
        if pages:
            if shared_len != len(pages) * self.page_size:
                raise PkvError(-1, "a shared prefix must fill whole pages")
            self.allocator.incref(pages)
        self.pages[rid] = pages
        self.lens[rid] = int(shared_len)

    def fork(self, src_rid: int, new_rid: int):
        """A new request sharing every page of ``src_rid`` (parallel sampling, beam search);
        writes into a shared, partly filled page first copy it (``reserve`` does that)."""
        if new_rid in self.pages:
            raise PkvError(-1, "request %d exists" % new_rid)
        pages = list(self.pages[src_rid])
        live = [p for p in pages if p >= 0]
        if live:
            self.allocator.incref(live)
        self.pages[new_rid] = pages
        self.lens[new_rid] = self.lens[src_rid]

    def free_request(self, rid: int):
        self.allocator.decref([p for p in self.pages.pop(rid) if p >= 0])
        del self.lens[rid]

    def release_outside_window(self, rid: int, window: int, sink_tokens: int = 0) -> int:
        """Sliding window ("KV cache and PagedAttention", section 8): return to the allocator
        every page of the request whose positions all lie outside the first ``sink_tokens``
        and the last ``window`` positions (the window only moves forward, so they are never
        read again). Their table entries become -1. Returns the number of pages released."""
        if window <= 0:
            return 0
        n, P = self.lens[rid], self.page_size
        pages = self.pages[rid]
        released = []
        for lp, pid in enumerate(pages):
            if pid < 0:
                continue
            first, last = lp * P, min(lp * P + P, n) - 1
            if last < n - 1 and first >= sink_tokens and last < n - window:
                released.append(pid)
                pages[lp] = -1
        if released:
            self.allocator.decref(released)
        return len(released)

    def reserve(self, rids, counts, copies_out=None) -> np.ndarray:
        """Grow each request by counts[i] tokens (allocating pages on page boundaries) and
        return the int64 slots of the new positions, request by request. Shared, partly filled
        pages about to be written are copied first (copy-on-write): on the device here, or,
        when ``copies_out`` is a list, appended to it as (source, destination) page pairs for
        the caller to copy (``copy_pages``) before the writes."""
        rids = list(rids)
        counts = [int(c) for c in counts]
        copies = []
        for rid, n in zip(rids, counts):
            if n > 0:  # copy-on-write of a shared, partly filled page before writing into it
                pair = self.allocator.cow_page(self.pages[rid], self.lens[rid], self.page_size)
                if pair is not None:
                    copies.append(pair)
            need = pages_needed(self.lens[rid] + n, self.page_size) - len(self.pages[rid])
            if need > 0:
                self.pages[rid].extend(int(p) for p in self.allocator.alloc(need))
        width = max([len(self.pages[r]) for r in rids] + [1])
        table = self.block_table_array(rids, width)
        total = sum(counts)
        req = np.empty(total, dtype=np.int32)
        pos = np.empty(total, dtype=np.int64)
        o = 0
        for i, (rid, n) in enumerate(zip(rids, counts)):
            req[o:o + n] = i
            pos[o:o + n] = np.arange(self.lens[rid], self.lens[rid] + n)
            o += n
            self.lens[rid] += n
        if copies_out is not None:
            copies_out.extend(copies)
        elif copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device=self.k.device)
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device=self.k.device)
            copy_pages(self.k, self.v, src, dst)
        return slot_mapping(table, pos, self.num_pages, requests=req, page_size=self.page_size)

    def write(self, slots, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Append rows k_new/v_new [N, h_kv, d] at the given slots (host array or CUDA int64)."""
        if not isinstance(slots, torch.Tensor):
            slots = torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(self.k.device)
        kv_append(k_new, v_new, slots, self.k, self.v, self.k_scales, self.v_scales, stream)

    # ---- views for the decode ---------------------------------------------------------------

    def block_table_array(self, rids, width: int | None = None) -> np.ndarray:
        rids = list(rids)
        if width is None:
            width = max([len(self.pages[r]) for r in rids] + [1])
        bt = np.zeros((len(rids), width), dtype=np.int32)
        for i, r in enumerate(rids):
            p = self.pages[r]
            bt[i, :len(p)] = p  # released pages stay as -1
        return bt

    def context_lens_array(self, rids) -> np.ndarray:
        return np.array([self.lens[r] for r in rids], dtype=np.int32)
