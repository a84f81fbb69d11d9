"""One layer's paged KV cache: the two pools plus the host bookkeeping around them.

"KV cache and PagedAttention", section 4: a physical pool of fixed-size pages and, per
request, a page table listing its pages; the allocator is O(1); requests with a common
prefix point at the same pages (reference-counted here). Section 5 (continuous batching):
requests join and leave the running batch every step, so pages are freed and reused.

Page accounting, the allocator and the per-request page tables (fork, free, reserve with
copy-on-write, window release, table export) run in the C library (``pkv_alloc``/``pkv_incref``/
``pkv_decref``, ``pkv_seq_*``); this class holds the pools and hands tensors to the kernels.
"""
from __future__ import annotations

from collections.abc import Mapping

import numpy as np
import torch

from . import PageAllocator, SeqTable, copy_pages, kv_append


class _RowView(Mapping):
    """Read-only view of the request table: rid -> page row (list) or token count (int)."""

    def __init__(self, table: SeqTable, what: str):
        self._t, self._what = table, what

    def __getitem__(self, rid):
        return self._t.pages(rid) if self._what == "pages" else self._t.length(rid)

    def __iter__(self):
        return iter(self._t.ids())

    def __len__(self):
        return len(self._t.ids())

    def __contains__(self, rid):
        try:
            self._t.length(rid)
        except KeyError:
            return False
        return True


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
        self.table = SeqTable(self.allocator, page_size)
        self.k_scales = k_scales
        self.v_scales = v_scales
        self.pages = _RowView(self.table, "pages")  # rid -> list of page ids (-1: released)
        self.lens = _RowView(self.table, "lens")    # rid -> tokens held

    @property
    def is_fp8(self) -> bool:
        return self.k.dtype == torch.uint8

    @property
    def is_int8(self) -> bool:
        return self.k.dtype == torch.int8

    # ---- requests ---------------------------------------------------------------------------

    def add_request(self, rid: int, shared_pages=None, shared_len: int = 0, adopt: bool = False):
        """New request; optionally starting on ``shared_pages`` that already hold its first
        ``shared_len`` tokens (a prefix, whole pages only). ``adopt``: the request takes over
        references the caller holds on those pages instead of taking new ones."""
        self.table.add(rid, shared_pages, shared_len, adopt)

    def add_request_from_prefix_cache(self, rid: int, prefix_cache, tenant: int, tokens) -> int:
        """New request whose prompt is ``tokens``: it starts on the longest prefix of whole
        pages that ``prefix_cache`` holds for this tenant (the lookup's references become the
        request's). Returns the number of prompt tokens already in the cache; the caller
        reserves and writes the rest."""
        return prefix_cache.add_request(self.table, rid, tenant, tokens)

    def register_prompt(self, rid: int, prefix_cache, tenant: int, tokens):
        """Puts the full pages of request ``rid``'s prompt (``tokens``, already written) into
        ``prefix_cache`` for later requests of the same tenant."""
        prefix_cache.insert_request(tenant, tokens, self.table, rid)

    def fork(self, src_rid: int, new_rid: int):
        """A new request sharing every page of ``src_rid`` (parallel sampling, beam search);
        writes into a shared, partly filled page first copy it (``reserve`` does that)."""
        self.table.fork([src_rid], [new_rid])

    def fork_many(self, src_rids, new_rids):
        """``fork`` for several requests in one call (a parent may be forked earlier in it)."""
        self.table.fork(src_rids, new_rids)

    def free_request(self, rid: int):
        self.table.free([rid])

    def free_many(self, rids):
        self.table.free(rids)

    def release_outside_window(self, rid: int, window: int, sink_tokens: int = 0) -> int:
        """Sliding window ("KV cache and PagedAttention", section 8): return to the allocator
        every page of the request whose positions all lie outside the first ``sink_tokens``
        and the last ``window`` positions (the window only moves forward, so they are never
        read again). Their table entries become -1. Returns the number of pages released."""
        return self.table.release_outside_window(rid, window, sink_tokens)

    def reserve(self, rids, counts, copies_out=None) -> np.ndarray:
        """Grow each request by counts[i] tokens (allocating pages on page boundaries) and
        return the int64 slots of the new positions, request by request. Shared, partly filled
        pages about to be written are copied first (copy-on-write): on the device here, or,
        when ``copies_out`` is a list, appended to it as (source, destination) page pairs for
        the caller to copy (``copy_pages``) before the writes."""
        slots, copies = self.table.reserve(rids, counts)
        if copies_out is not None:
            copies_out.extend(copies)
        elif copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device=self.k.device)
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device=self.k.device)
            copy_pages(self.k, self.v, src, dst)
        return slots

    def step(self, finished, joining, prompt_lens, live, width: int | None = None,
             tables_out=None, lens_out=None, copies_out=None, incremental: bool = False):
        """One continuous-batching step of bookkeeping in one library call: the ``finished``
        requests are freed, the ``joining`` ones added and grown by their ``prompt_lens``, every
        ``live`` request (joining ones included) gets room for one new token, and the live
        requests' page-table rows and lengths are exported (into ``tables_out``/``lens_out``
        when given). Returns (prompt slots, tables, lengths). Shared pages about to be written
        are copied as in ``reserve``. If the pages run out, the frees stand and the joining
        requests are not added (PkvError). ``incremental``: rows of ``tables_out`` that still
        hold the same request as after the previous incremental step are only patched."""
        slots, bt, cl, copies = self.table.step(finished, joining, prompt_lens, live, width,
                                                tables_out, lens_out, incremental=incremental)
        if copies_out is not None:
            copies_out.extend(copies)
        elif copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device=self.k.device)
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device=self.k.device)
            copy_pages(self.k, self.v, src, dst)
        return slots, bt, cl

    def write(self, slots, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Append rows k_new/v_new [N, h_kv, d] at the given slots (host array or CUDA int64)."""
        if not isinstance(slots, torch.Tensor):
            slots = torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(self.k.device)
        kv_append(k_new, v_new, slots, self.k, self.v, self.k_scales, self.v_scales, stream)

    # ---- views for the decode ---------------------------------------------------------------

    def block_table_array(self, rids, width: int | None = None, out=None) -> np.ndarray:
        """Page-table rows of the requests (unused columns 0, released pages -1); ``out`` (a
        contiguous int32 array or CPU tensor of [len(rids)][width]) is filled in place."""
        return self.table.tables(rids, width, out=out)

    def context_lens_array(self, rids, out=None) -> np.ndarray:
        return self.table.lengths(rids, out=out)
