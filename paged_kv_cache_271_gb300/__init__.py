"""Paged KV cache for single-token decode attention on GB300 (sm_103a).

A thin ctypes binding over ``libpkv.so`` (C ABI declared in ``include/pkv.h``): argument
marshalling only, every step of the decode path runs in the library's CUDA kernels. torch
supplies device memory and streams. The library must have been built (``python -m
paged_kv_cache_271_gb300.build``); calls fail loudly otherwise -- there is no fallback.

Entry points (same names as the C ABI, without the ``pkv_`` prefix):
``kv_append``, ``paged_decode_attention``, ``decode_workspace_size``, ``kv_absmax_scales``,
``device_error``, ``pages_needed``, ``slot_mapping``, ``PageAllocator`` (``pkv_alloc``,
``pkv_incref``, ``pkv_decref``, ...), ``PrefixCache`` (``pkv_prefix_*``), ``cascade_groups``,
``cascade_decode_attention``, ``cascade_decode_step``, ``decode_set_chunk_pages``, ``trace_*``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

__all__ = [
    "PkvError", "F32", "BF16", "FP8_E4M3", "lib", "library_path", "cache_desc", "kv_append",
    "decode_workspace_size", "paged_decode_attention", "kv_absmax_scales", "device_error",
    "decode_set_chunk_pages", "decode_chunk_pages", "pages_needed", "slot_mapping",
    "PageAllocator", "PrefixCache", "CascadeGroups", "cascade_groups", "cascade_decode_attention",
    "cascade_decode_step", "cascade_workspace_size", "HostStep", "trace_enable", "trace_reset",
    "trace_read",
]

F32, BF16, FP8_E4M3, INT8 = 0, 1, 2, 3
DEVERR_BAD_PAGE, DEVERR_BAD_SLOT, DEVERR_TIMEOUT, DEVERR_BAD_GROUP = 1, 2, 4, 8
_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpkv.so")
_lib = None


class PkvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("pkv error %d: %s" % (code, msg))
        self.code = code


class _Desc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32)]


class _CascadeDesc(ctypes.Structure):
    _fields_ = [("group_of", ctypes.c_void_p), ("prefix_pages", ctypes.c_void_p),
                ("group_offsets", ctypes.c_void_p), ("group_members", ctypes.c_void_p),
                ("n_groups", ctypes.c_int32), ("max_members", ctypes.c_int32),
                ("max_prefix_pages", ctypes.c_int32), ("max_own_pages", ctypes.c_int32),
                ("own_start", ctypes.c_void_p), ("prefix_page_ids", ctypes.c_void_p)]


def lib():
    """The loaded C library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError("libpkv.so is not built (run `python -m paged_kv_cache_271_gb300.build`"
                           " or __graft_entry__.build()); there is no fallback path")
    L = ctypes.CDLL(library_path)
    vp, i32, i64, f32, dbl, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
    D = ctypes.POINTER(_Desc)
    C = ctypes.POINTER(_CascadeDesc)
    sig = {
        "pkv_last_error": (ctypes.c_char_p, []),
        "pkv_version": (ctypes.c_int, []),
        "pkv_kv_append": (ctypes.c_int, [vp, vp, i32, i32, vp, vp, vp, D, vp, vp, vp]),
        "pkv_decode_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "pkv_paged_decode_attention": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, D, vp, i32, vp,
                                                      f32, vp, vp, vp, vp, sz, vp]),
        "pkv_paged_decode_step": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, i32, vp, vp, D, vp,
                                                 i32, vp, f32, vp, vp, vp, vp, sz, vp]),
        "pkv_paged_decode_attention_window": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, D, vp,
                                                             i32, vp, f32, vp, vp, i32, i32, vp,
                                                             vp, sz, vp]),
        "pkv_paged_decode_step_window": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, i32, vp, vp, D,
                                                        vp, i32, vp, f32, vp, vp, i32, i32, vp,
                                                        vp, sz, vp]),
        "pkv_paged_decode_attention_noalloc": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, D, vp,
                                                              i32, vp, f32, vp, vp, vp, vp]),
        "pkv_decode_noalloc_scratch_bytes": (sz, []),
        "pkv_kv_absmax_scales": (ctypes.c_int, [vp, i32, i64, i32, i32, vp, vp]),
        "pkv_kv_absmax_scales_int8": (ctypes.c_int, [vp, i32, i64, i32, i32, vp, vp]),
        "pkv_device_error": (ctypes.c_int, [vp, ctypes.POINTER(i32)]),
        "pkv_decode_set_chunk_pages": (ctypes.c_int, [i32]),
        "pkv_decode_chunk_pages": (i32, [i32, i32, i32]),
        "pkv_decode_set_kernel": (ctypes.c_int, [i32]),
        "pkv_decode_set_split": (ctypes.c_int, [i32]),
        "pkv_decode_set_autotune": (ctypes.c_int, [i32]),
        "pkv_decode_autotune_reset": (ctypes.c_int, []),
        "pkv_decode_split_choice": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32, i32, i32]),
        "pkv_decode_set_merge_in_place": (ctypes.c_int, [i32]),
        "pkv_decode_set_warp_per_request": (ctypes.c_int, [i32]),
        "pkv_cascade_set_overlap": (ctypes.c_int, [i32]),
        "pkv_pages_needed": (ctypes.c_int, [i64, i32, ctypes.POINTER(i64)]),
        "pkv_slot_mapping": (ctypes.c_int, [vp, i32, vp, vp, i64, i32, i32, vp]),
        "pkv_allocator_create": (ctypes.c_int, [i32, vp, ctypes.POINTER(vp)]),
        "pkv_allocator_destroy": (None, [vp]),
        "pkv_alloc": (ctypes.c_int, [vp, i32, vp]),
        "pkv_incref": (ctypes.c_int, [vp, vp, i32]),
        "pkv_decref": (ctypes.c_int, [vp, vp, i32]),
        "pkv_num_free": (i32, [vp]),
        "pkv_cow_page": (ctypes.c_int, [vp, vp, i32, i64, i32, ctypes.POINTER(i32),
                                        ctypes.POINTER(i32)]),
        "pkv_copy_pages": (ctypes.c_int, [vp, vp, D, vp, vp, i32, vp]),
        "pkv_refcount": (i32, [vp, i32]),
        "pkv_seq_table_create": (ctypes.c_int, [vp, i32, ctypes.POINTER(vp)]),
        "pkv_seq_table_destroy": (None, [vp]),
        "pkv_seq_add": (ctypes.c_int, [vp, i64, vp, i32, i64]),
        "pkv_seq_adopt": (ctypes.c_int, [vp, i64, vp, i32, i64]),
        "pkv_seq_fork": (ctypes.c_int, [vp, vp, vp, i32]),
        "pkv_seq_free": (ctypes.c_int, [vp, vp, i32]),
        "pkv_seq_reserve": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, vp, ctypes.POINTER(i32)]),
        "pkv_seq_tables": (ctypes.c_int, [vp, vp, i32, i32, vp, vp]),
        "pkv_seq_step": (ctypes.c_int, [vp, vp, i32, vp, vp, i32, vp, vp, i32, vp, i32, vp, vp,
                                        i32, vp, vp, ctypes.POINTER(i32)]),
        "pkv_seq_step_width": (ctypes.c_int, [vp, vp, vp, i32, vp, i32, ctypes.POINTER(i32)]),
        "pkv_seq_add_cached_prefix": (ctypes.c_int, [vp, i64, vp, i64, vp, i64,
                                                     ctypes.POINTER(i64)]),
        "pkv_prefix_insert_request": (ctypes.c_int, [vp, i64, vp, i64, vp, i64]),
        "pkv_seq_release_outside_window": (ctypes.c_int, [vp, i64, i64, i64,
                                                          ctypes.POINTER(i32)]),
        "pkv_seq_len": (i64, [vp, i64]),
        "pkv_seq_pages": (i32, [vp, i64, vp, i32]),
        "pkv_seq_count": (i32, [vp]),
        "pkv_seq_ids": (i32, [vp, vp, i32]),
        "pkv_prefix_cache_create": (ctypes.c_int, [vp, i32, ctypes.POINTER(vp)]),
        "pkv_prefix_cache_destroy": (None, [vp]),
        "pkv_prefix_lookup": (ctypes.c_int, [vp, i64, vp, i64, vp, i32, ctypes.POINTER(i32)]),
        "pkv_prefix_insert": (ctypes.c_int, [vp, i64, vp, i64, vp, i32]),
        "pkv_prefix_evict": (ctypes.c_int, [vp, i32, ctypes.POINTER(i32)]),
        "pkv_prefix_size": (i32, [vp]),
        "pkv_packed_step_layout": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32, vp,
                                                  ctypes.POINTER(sz)]),
        "pkv_paged_decode_step_packed": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, D, i32,
                                                        f32, vp, vp, i32, i32, vp, vp, vp, sz,
                                                        vp]),
        "pkv_packed_cascade_layout": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32, vp,
                                                     ctypes.POINTER(sz)]),
        "pkv_cascade_decode_step_packed": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, D,
                                                          i32, f32, vp, vp, vp, sz,
                                                          ctypes.POINTER(sz), ctypes.POINTER(i32),
                                                          vp]),
        "pkv_cascade_groups": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp,
                                              ctypes.POINTER(i32), ctypes.POINTER(i32),
                                              ctypes.POINTER(i32), ctypes.POINTER(i32), vp]),
        "pkv_cascade_workspace_size": (sz, [i32, i32, i32, i32, i32, C]),
        "pkv_cascade_prefix_page_ids": (ctypes.c_int, [vp, i32, i32, vp, vp, vp, i32, i32, vp]),
        "pkv_cascade_prefix_chunk_pages": (i32, [i32, i32, C]),
        "pkv_cascade_decode_attention": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, D, vp, i32,
                                                        vp, f32, C, vp, vp, sz, vp]),
        "pkv_cascade_decode_step": (ctypes.c_int, [vp, i32, i32, i32, vp, vp, i32, vp, vp, D, vp,
                                                   i32, vp, f32, C, vp, vp, sz, vp]),
        "pkv_cascade_set_prefix_chunk_pages": (ctypes.c_int, [i32]),
        "pkv_cascade_set_prefix_kernel": (ctypes.c_int, [i32]),
        "pkv_trace_enable": (ctypes.c_int, [ctypes.c_int]),
        "pkv_trace_reset": (ctypes.c_int, []),
        "pkv_selftest_wait_timeout": (ctypes.c_int, [vp, vp, vp]),
        "pkv_trace_read": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(i32),
                                          ctypes.POINTER(dbl)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(st: int):
    if st != 0:
        raise PkvError(st, lib().pkv_last_error().decode())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    if t.dtype == torch.int8:
        return INT8
    raise PkvError(-3, "unsupported dtype %s" % t.dtype)


def _dev(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise PkvError(-1, "%s must be a CUDA tensor" % name)
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device, whose kernels cannot read another GPU's
        # memory without peer access
        raise PkvError(-1, "%s is on %s but the current device is cuda:%d" %
                       (name, t.device, torch.cuda.current_device()))
    if not t.is_contiguous():
        raise PkvError(-1, "%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _opt(t, name):
    return None if t is None else _dev(t, name)


def cache_desc(k_cache: torch.Tensor) -> _Desc:
    """Descriptor of a pool [num_pages, num_kv_heads, page_size, head_dim]; uint8 or
    float8_e4m3fn pools are FP8 E4M3 caches, int8 pools INT8 caches."""
    if k_cache.dim() != 4:
        raise PkvError(-2, "pool must be [num_pages, num_kv_heads, page_size, head_dim]")
    n, h, p, d = k_cache.shape
    return _Desc(n, p, h, d, _dtype_code(k_cache))


def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, k_scales=None, v_scales=None,
              stream=None):
    """Write phase: k_new/v_new [N, h_kv, d] into the pools at slot_mapping (int64 [N])."""
    if slot_mapping.dtype != torch.int64:
        raise PkvError(-3, "slot_mapping must be int64")
    if k_new.shape != v_new.shape or k_new.dim() != 3:
        raise PkvError(-2, "k_new and v_new must both be [N, h_kv, d]")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise PkvError(-2, "k_cache and v_cache differ")
    if slot_mapping.numel() != k_new.shape[0]:
        raise PkvError(-2, "slot_mapping length != number of tokens")
    desc = cache_desc(k_cache)
    if k_new.shape[1] != desc.num_kv_heads or k_new.shape[2] != desc.head_dim:
        raise PkvError(-2, "k_new heads/dims do not match the pool")
    _check(lib().pkv_kv_append(_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dtype_code(k_new),
                               k_new.shape[0], _dev(slot_mapping, "slot_mapping"),
                               _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                               ctypes.byref(desc), _opt(k_scales, "k_scales"),
                               _opt(v_scales, "v_scales"), _stream(stream)))


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_pages_per_seq) -> int:
    return int(lib().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                               max_pages_per_seq))


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                           k_scales=None, v_scales=None, workspace=None, stream=None, window=0,
                           sink_tokens=0):
    """Read phase: decode attention of q [B, h_q, d] over the paged pools; returns out.
    window > 0: attend only the last ``window`` positions plus the first ``sink_tokens``
    (pkv_paged_decode_attention_window)."""
    if q.dim() != 3:
        raise PkvError(-2, "q must be [batch, num_q_heads, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError(-3, "block_tables and context_lens must be int32")
    B, h_q, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise PkvError(-2, "block_tables must be [batch, max_pages], context_lens [batch]")
    desc = cache_desc(k_cache)
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise PkvError(-2, "k_cache and v_cache differ")
    if d != desc.head_dim:
        raise PkvError(-2, "q head_dim does not match the pool")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype:
        raise PkvError(-2, "out must match q in shape and dtype")
    maxp = block_tables.shape[1]
    need = decode_workspace_size(B, h_q, desc.num_kv_heads, d, maxp)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws = _opt(workspace, "workspace")
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_dev(q, "q"), _dtype_code(q), B, h_q, _dev(k_cache, "k_cache"),
            _dev(v_cache, "v_cache"), ctypes.byref(desc), _dev(block_tables, "block_tables"), maxp,
            _dev(context_lens, "context_lens"), float(scale), _opt(k_scales, "k_scales"),
            _opt(v_scales, "v_scales")]
    tail = [_dev(out, "out"), ws, wsb, _stream(stream)]
    if window or sink_tokens:
        _check(lib().pkv_paged_decode_attention_window(*args, int(sink_tokens), int(window),
                                                       *tail))
    else:
        _check(lib().pkv_paged_decode_attention(*args, *tail))
    return out


def paged_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                      out=None, k_scales=None, v_scales=None, workspace=None, stream=None,
                      window=0, sink_tokens=0):
    """Append + decode in one launch: k_new/v_new [B, h_kv, d] go to position
    context_lens[b] - 1 of each request, then attention over positions 0 .. context_lens[b]-1.
    A workspace, when needed, must be zero-filled before its first use (allocated zeroed here
    when not given)."""
    if q.dim() != 3 or k_new.dim() != 3 or k_new.shape != v_new.shape:
        raise PkvError(-2, "q must be [B, h_q, d], k_new and v_new [B, h_kv, d]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError(-3, "block_tables and context_lens must be int32")
    B, h_q, d = q.shape
    desc = cache_desc(k_cache)
    if k_new.shape[0] != B or k_new.shape[1] != desc.num_kv_heads or k_new.shape[2] != d:
        raise PkvError(-2, "k_new must be [batch, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    maxp = block_tables.shape[1]
    need = decode_workspace_size(B, h_q, desc.num_kv_heads, d, maxp)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_dev(q, "q"), _dtype_code(q), B, h_q, _dev(k_new, "k_new"), _dev(v_new, "v_new"),
            _dtype_code(k_new), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            ctypes.byref(desc), _dev(block_tables, "block_tables"), maxp,
            _dev(context_lens, "context_lens"), float(scale), _opt(k_scales, "k_scales"),
            _opt(v_scales, "v_scales")]
    tail = [_dev(out, "out"), _opt(workspace, "workspace"), wsb, _stream(stream)]
    if window or sink_tokens:
        _check(lib().pkv_paged_decode_step_window(*args, int(sink_tokens), int(window), *tail))
    else:
        _check(lib().pkv_paged_decode_step(*args, *tail))
    return out


class CascadeGroups:
    """Groups of a batch that share leading pages (pkv_cascade_groups), as host arrays; call
    ``to(device)`` once to place them for the cascade decode."""

    def __init__(self, group_of, prefix_pages, group_offsets, group_members, max_members,
                 max_prefix_pages, max_own_pages=0, own_start=None, prefix_page_ids=None):
        self.group_of = group_of
        self.prefix_pages = prefix_pages
        self.group_offsets = group_offsets
        self.group_members = group_members
        self.n_groups = len(prefix_pages)
        self.max_members = int(max_members)
        self.max_prefix_pages = int(max_prefix_pages)
        self.max_own_pages = int(max_own_pages)
        if own_start is None:  # prefix_pages[group_of[b]], 0 outside a group
            own_start = np.where(group_of >= 0, np.append(prefix_pages, 0)[group_of], 0)
        self.own_start = np.asarray(own_start, dtype=np.int32)
        # [n_groups][max_prefix_pages] shared page ids (pkv_cascade_prefix_page_ids), or None
        self.prefix_page_ids = (None if prefix_page_ids is None else
                                np.asarray(prefix_page_ids, dtype=np.int32).reshape(-1))
        self._dev = None

    def packed(self) -> np.ndarray:
        """The arrays back to back (int32), as ``to`` places them."""
        parts = [self.group_of, self.prefix_pages, self.group_offsets, self.group_members,
                 self.own_start]
        if self.prefix_page_ids is not None:
            parts.append(self.prefix_page_ids)
        return np.concatenate(parts).astype(np.int32)

    def to(self, device, buffer=None, staging=None):
        """Place the arrays on the device in one copy: into a new tensor, or into ``buffer``
        (int32 device tensor) through ``staging`` (pinned int32 host tensor), asynchronously."""
        p = self.packed()
        if buffer is None:
            buffer = torch.from_numpy(p).to(device)
        else:
            if buffer.numel() < p.size or staging is None or staging.numel() < p.size:
                raise PkvError(-1, "cascade group buffers are too small")
            staging[:p.size].copy_(torch.from_numpy(p))
            buffer[:p.size].copy_(staging[:p.size], non_blocking=True)
        self._dev = buffer
        self.nbytes = 4 * p.size
        B, ng, nm = len(self.group_of), self.n_groups, len(self.group_members)
        base = buffer.data_ptr()
        self._ptrs = [base, base + 4 * B, base + 4 * (B + ng), base + 4 * (B + 2 * ng + 1),
                      base + 4 * (B + 2 * ng + 1 + nm)]
        self._ids_ptr = (None if self.prefix_page_ids is None else
                         base + 4 * (2 * B + 2 * ng + 1 + nm))
        return self

    def desc(self) -> _CascadeDesc:
        if self.n_groups == 0:
            return _CascadeDesc(None, None, None, None, 0, 0, 0)
        if self._dev is None:
            raise PkvError(-1, "CascadeGroups.to(device) has not been called")
        g, p, o, m, st = self._ptrs
        return _CascadeDesc(g, p, o, m, self.n_groups, self.max_members, self.max_prefix_pages,
                            self.max_own_pages, st, self._ids_ptr)


def cascade_groups(block_tables, context_lens, min_members=2, min_prefix_pages=1) -> CascadeGroups:
    """Requests whose tables start with the same pages (host arrays; pkv_cascade_groups)."""
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    B, W = bt.shape
    if cl.shape != (B,):
        raise PkvError(-2, "context_lens must be [batch]")
    group_of = np.empty(B, np.int32)
    prefix = np.empty(max(B, 1), np.int32)
    offs = np.empty(B + 1, np.int32)
    members = np.empty(max(B, 1), np.int32)
    n, mm, mp, mo = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    start = np.empty(max(B, 1), np.int32)
    _check(lib().pkv_cascade_groups(bt.ctypes.data if B else None, cl.ctypes.data if B else None,
                                    B, W, int(min_members), int(min_prefix_pages),
                                    group_of.ctypes.data, prefix.ctypes.data, offs.ctypes.data,
                                    members.ctypes.data, ctypes.byref(n), ctypes.byref(mm),
                                    ctypes.byref(mp), ctypes.byref(mo), start.ctypes.data))
    ng = n.value
    ids = np.empty(max(ng * mp.value, 1), np.int32)
    if ng:
        _check(lib().pkv_cascade_prefix_page_ids(bt.ctypes.data, B, W, prefix.ctypes.data,
                                                 offs.ctypes.data, members.ctypes.data, ng,
                                                 mp.value, ids.ctypes.data))
    return CascadeGroups(group_of, prefix[:ng].copy(), offs[:ng + 1].copy(),
                         members[:offs[ng]].copy(), mm.value, mp.value, mo.value, start[:B].copy(),
                         ids[:ng * mp.value].copy() if ng else None)


def cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_pages_per_seq,
                           groups: CascadeGroups) -> int:
    d = groups.desc() if groups.n_groups == 0 or groups._dev is not None else _CascadeDesc(
        None, None, None, None, groups.n_groups, groups.max_members, groups.max_prefix_pages,
        groups.max_own_pages)
    return int(lib().pkv_cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                max_pages_per_seq, ctypes.byref(d)))


def cascade_prefix_chunk_pages(num_kv_heads, num_q_heads, groups: CascadeGroups) -> int:
    d = _CascadeDesc(None, None, None, None, groups.n_groups, groups.max_members,
                     groups.max_prefix_pages)
    return int(lib().pkv_cascade_prefix_chunk_pages(num_kv_heads, num_q_heads, ctypes.byref(d)))


def cascade_set_prefix_chunk_pages(pages: int):
    _check(lib().pkv_cascade_set_prefix_chunk_pages(int(pages)))


def cascade_set_prefix_kernel(which: int):
    """0 automatic (tcgen05), 1 mma.sync, 2 tcgen05."""
    _check(lib().pkv_cascade_set_prefix_kernel(int(which)))


def _cascade_common(q, k_cache, block_tables, context_lens, groups, workspace):
    if q.dim() != 3 or block_tables.dim() != 2:
        raise PkvError(-2, "q must be [batch, heads, dim], block_tables [batch, max_pages]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError(-3, "block_tables and context_lens must be int32")
    B, h_q, d = q.shape
    desc = cache_desc(k_cache)
    maxp = block_tables.shape[1]
    need = cascade_workspace_size(B, h_q, desc.num_kv_heads, d, maxp, groups)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return B, h_q, desc, maxp, workspace, wsb


def cascade_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                             groups: CascadeGroups, out=None, workspace=None, stream=None):
    """Decode attention with each group's shared pages computed once for all its members
    (pkv_cascade_decode_attention); same result as paged_decode_attention."""
    B, h_q, desc, maxp, workspace, wsb = _cascade_common(q, k_cache, block_tables, context_lens,
                                                         groups, workspace)
    if out is None:
        out = torch.empty_like(q)
    gd = groups.desc()
    _check(lib().pkv_cascade_decode_attention(
        _dev(q, "q"), _dtype_code(q), B, h_q, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        ctypes.byref(desc), _dev(block_tables, "block_tables"), maxp,
        _dev(context_lens, "context_lens"), float(scale), ctypes.byref(gd), _dev(out, "out"),
        _opt(workspace, "workspace"), wsb, _stream(stream)))
    return out


def cascade_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                        groups: CascadeGroups, out=None, workspace=None, stream=None):
    """paged_decode_step with each group's shared pages computed once (pkv_cascade_decode_step)."""
    B, h_q, desc, maxp, workspace, wsb = _cascade_common(q, k_cache, block_tables, context_lens,
                                                         groups, workspace)
    if k_new.shape != v_new.shape or k_new.dim() != 3 or k_new.shape[0] != B:
        raise PkvError(-2, "k_new and v_new must both be [batch, h_kv, d]")
    if out is None:
        out = torch.empty_like(q)
    gd = groups.desc()
    _check(lib().pkv_cascade_decode_step(
        _dev(q, "q"), _dtype_code(q), B, h_q, _dev(k_new, "k_new"), _dev(v_new, "v_new"),
        _dtype_code(k_new), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        ctypes.byref(desc), _dev(block_tables, "block_tables"), maxp,
        _dev(context_lens, "context_lens"), float(scale), ctypes.byref(gd), _dev(out, "out"),
        _opt(workspace, "workspace"), wsb, _stream(stream)))
    return out


class HostStep:
    """A decode step whose inputs live in host memory: the step's queries, new K/V rows, page
    tables and context lengths are packed into one pinned buffer (the ``*_host`` views, filled
    by the caller, laid out by pkv_packed_step_layout); ``step`` makes one library call
    (pkv_paged_decode_step_packed) that copies them to the device, runs the fused append +
    decode (windowed when ``window`` > 0) and copies the output into ``out_host``. With
    ``use_graph`` that call is captured once per set of call arguments (pools, workspace,
    stream, scale, window) as a CUDA graph, and later steps replay it: the same two copies and
    kernels, read from and written to the same pinned buffers, for one launch. The first step
    of each new set runs the call once before capturing it (the fused append rewrites the same
    row, so the repeat changes nothing). It is off by default: on a GB300 the replayed step,
    host copies included, measured slower than the call made op by op (Llama-3-8B batch 64:
    138.8 vs 129.1 us). With cascade ``groups`` (whose arrays change the launch) the copies are
    made here and the step is cascade_decode_step."""

    _CODE = {torch.float32: F32, torch.bfloat16: BF16}

    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, max_pages,
                 q_dtype=torch.bfloat16, new_dtype=torch.bfloat16, device="cuda",
                 use_graph=False, cascade=False):
        self.use_graph = bool(use_graph)
        self.cascade = bool(cascade)  # room for the groups (cascade_step)
        self._graphs = {}
        self.batch, self.h_q, self.max_pages = batch, num_q_heads, max_pages
        self.q_code, self.new_code = self._CODE[q_dtype], self._CODE[new_dtype]
        offs = (ctypes.c_size_t * 11)()
        total = ctypes.c_size_t(0)
        layout = lib().pkv_packed_cascade_layout if cascade else lib().pkv_packed_step_layout
        _check(layout(batch, num_q_heads, num_kv_heads, head_dim, max_pages, self.q_code,
                      self.new_code, offs, ctypes.byref(total)))
        self.h2d_bytes = int(total.value)
        self.host = torch.empty(self.h2d_bytes, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(self.h2d_bytes, dtype=torch.uint8, device=device)
        parts = [("q", (batch, num_q_heads, head_dim), q_dtype),
                 ("k_new", (batch, num_kv_heads, head_dim), new_dtype),
                 ("v_new", (batch, num_kv_heads, head_dim), new_dtype),
                 ("block_tables", (batch, max_pages), torch.int32),
                 ("context_lens", (batch,), torch.int32)]
        for (name, shape, dt), o in zip(parts, offs):
            n = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
            setattr(self, name + "_host", self.host[o:o + n].view(dt).view(shape))
            setattr(self, name, self.dev[o:o + n].view(dt).view(shape))
        self.out = torch.empty((batch, num_q_heads, head_dim), dtype=q_dtype, device=device)
        self.out_host = torch.empty(self.out.shape, dtype=q_dtype).pin_memory()
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        self._key = None
        self.n_groups = 0
        self.workspace_needed = 0

    def step(self, k_cache, v_cache, scale, k_scales=None, v_scales=None, workspace=None,
             groups=None, stream=None, window=0, sink_tokens=0):
        """One step; returns ``out_host`` (valid once the stream has reached this point)."""
        if groups is not None:
            st = torch.cuda.current_stream() if stream is None else stream
            with torch.cuda.stream(st):
                self.dev.copy_(self.host, non_blocking=True)
                cascade_decode_step(self.q, self.k_new, self.v_new, k_cache, v_cache,
                                    self.block_tables, self.context_lens, scale, groups,
                                    out=self.out, workspace=workspace, stream=st)
                self.out_host.copy_(self.out, non_blocking=True)
            return self.out_host
        sp = _stream(stream)
        key = (k_cache.data_ptr(), v_cache.data_ptr(), k_cache.shape, k_cache.stride(),
               v_cache.stride(), k_cache.dtype, float(scale),
               None if k_scales is None else k_scales.data_ptr(),
               None if v_scales is None else v_scales.data_ptr(),
               None if workspace is None else workspace.data_ptr(),
               None if workspace is None else workspace.numel() * workspace.element_size(),
               sp.value, int(window), int(sink_tokens))
        if key != self._key:  # the call's arguments, built once per pool / workspace / stream
            if workspace is None:
                need = decode_workspace_size(self.batch, self.h_q, k_cache.shape[1],
                                             k_cache.shape[3], self.max_pages)
                workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=self.dev.device)
            self._ws = workspace
            self._desc = cache_desc(k_cache)
            self._pre = (ctypes.c_void_p(self.host.data_ptr()), ctypes.c_void_p(self.dev.data_ptr()),
                         self.batch, self.h_q, self.q_code, self.new_code, _dev(k_cache, "k_cache"),
                         _dev(v_cache, "v_cache"), ctypes.byref(self._desc), self.max_pages,
                         float(scale), _opt(k_scales, "k_scales"), _opt(v_scales, "v_scales"),
                         int(sink_tokens), int(window), ctypes.c_void_p(self.out.data_ptr()),
                         ctypes.c_void_p(self.out_host.data_ptr()), _opt(workspace, "workspace"),
                         workspace.numel() * workspace.element_size())
            self._key = key
        if not self.use_graph:
            _check(lib().pkv_paged_decode_step_packed(*self._pre, sp))
            return self.out_host
        g = self._graphs.get(key)
        if stream is None:
            target = torch.cuda.current_stream(self.dev.device)
        elif isinstance(stream, torch.cuda.Stream):
            target = stream
        else:  # a raw cudaStream_t handle
            target = torch.cuda.ExternalStream(int(stream), device=self.dev.device)
        if g is None:
            side = torch.cuda.Stream(device=self.dev.device)
            side.wait_stream(target)
            _check(lib().pkv_paged_decode_step_packed(*self._pre, _stream(side)))  # warm-up
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                _check(lib().pkv_paged_decode_step_packed(*self._pre, _stream(side)))
            target.wait_stream(side)
            self._graphs[key] = g
        with torch.cuda.stream(target):
            g.replay()
        return self.out_host


    def cascade_step(self, k_cache, v_cache, scale, workspace, stream=None):
        """One cascade step from host memory (HostStep built with cascade=True): the library
        groups the batch from ``block_tables_host``/``context_lens_host``, copies the block once,
        runs the cascade (or, with no group, the plain) fused step and copies the output into
        ``out_host``. The workspace must hold ``workspace_needed`` bytes (set by every call; a
        first call with too small a workspace raises before anything is enqueued)."""
        if not self.cascade:
            raise PkvError(-1, "HostStep was built without cascade=True")
        wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
        key = (k_cache.data_ptr(), v_cache.data_ptr(), k_cache.shape, k_cache.stride(),
               v_cache.stride(), k_cache.dtype, float(scale),
               None if workspace is None else workspace.data_ptr(), wsb)
        if key != getattr(self, "_ckey", None):  # the call's arguments, built once per set
            self._cdesc = cache_desc(k_cache)
            self._need, self._ng = ctypes.c_size_t(0), ctypes.c_int32(0)
            self._cws = workspace
            self._cpre = (ctypes.c_void_p(self.host.data_ptr()), ctypes.c_void_p(self.dev.data_ptr()),
                          self.batch, self.h_q, self.q_code, self.new_code,
                          _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                          ctypes.byref(self._cdesc), self.max_pages, float(scale),
                          ctypes.c_void_p(self.out.data_ptr()),
                          ctypes.c_void_p(self.out_host.data_ptr()), _opt(workspace, "workspace"),
                          wsb, ctypes.byref(self._need), ctypes.byref(self._ng))
            self._ckey = key
        st = lib().pkv_cascade_decode_step_packed(*self._cpre, _stream(stream))
        self.workspace_needed = int(self._need.value)
        self.n_groups = int(self._ng.value)
        _check(st)
        return self.out_host

def paged_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale,
                                   out=None, k_scales=None, v_scales=None, stream=None):
    """paged_decode_attention without a workspace: for callers that cannot allocate device
    memory, the split partials go to the library's built-in 16 MiB scratch (shared by all calls
    on a device; calls that overlap on the GPU race)."""
    if q.dim() != 3 or block_tables.dim() != 2:
        raise PkvError(-2, "q must be [batch, heads, dim], block_tables [batch, max_pages]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError(-3, "block_tables and context_lens must be int32")
    B, h_q, _ = q.shape
    desc = cache_desc(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _check(lib().pkv_paged_decode_attention_noalloc(
        _dev(q, "q"), _dtype_code(q), B, h_q, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        ctypes.byref(desc), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), float(scale), _opt(k_scales, "k_scales"),
        _opt(v_scales, "v_scales"), _dev(out, "out"), _stream(stream)))
    return out


def copy_pages(k_cache, v_cache, src_pages, dst_pages, stream=None):
    """pool[dst_pages[p]] = pool[src_pages[p]] for both pools (device int32 id tensors)."""
    if src_pages.dtype != torch.int32 or dst_pages.dtype != torch.int32:
        raise PkvError(-3, "page ids must be int32")
    if src_pages.numel() != dst_pages.numel():
        raise PkvError(-2, "src_pages and dst_pages differ in length")
    desc = cache_desc(k_cache)
    _check(lib().pkv_copy_pages(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                ctypes.byref(desc), _dev(src_pages, "src_pages"),
                                _dev(dst_pages, "dst_pages"), src_pages.numel(), _stream(stream)))


def kv_absmax_scales(x, scales_out=None, stream=None, int8=False):
    """Scales per KV head: fp32(max|x[:, h, :]| / 448) for an FP8 cache, / 127 for an INT8
    cache (int8=True); 1 for an all-zero head."""
    if x.dim() != 3:
        raise PkvError(-2, "x must be [tokens, h_kv, d]")
    n, h, d = x.shape
    if scales_out is None:
        scales_out = torch.empty(h, dtype=torch.float32, device=x.device)
    fn = lib().pkv_kv_absmax_scales_int8 if int8 else lib().pkv_kv_absmax_scales
    _check(fn(_dev(x, "x"), _dtype_code(x), n, h, d, _dev(scales_out, "scales_out"),
              _stream(stream)))
    return scales_out


def device_error(stream=None) -> int:
    """Synchronise, then read and clear the device error word (0 when clean)."""
    code = ctypes.c_int32(0)
    st = lib().pkv_device_error(_stream(stream), ctypes.byref(code))
    if st not in (0, -8):
        _check(st)
    return int(code.value)


def decode_set_warp_per_request(on: bool):
    """One warp per request when every request fits one chunk of at most 16 pages (default)."""
    _check(lib().pkv_decode_set_warp_per_request(1 if on else 0))


def selftest_wait_timeout(stream=None):
    """Makes one bounded kernel wait run out on purpose (pkv_selftest_wait_timeout: a barrier
    nothing completes, given up after the kernels' 2 s limit) and returns (status bits, done):
    DEVERR_TIMEOUT set and done == 1 when the wait gave up as it should."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = torch.zeros_like(err)
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib().pkv_selftest_wait_timeout(_dev(err, "err"), _dev(done, "done"), _stream(st)))
    st.synchronize()
    return int(err.item()), int(done.item())


def cascade_set_overlap(on):
    """Cascade decode: run the own-page decode alongside the prefix kernel with the fold left
    to the combine kernel (2, the default), alongside it folding itself (True or 1), or after
    it (False or 0)."""
    _check(lib().pkv_cascade_set_overlap(int(on)))


def decode_set_chunk_pages(pages: int):
    _check(lib().pkv_decode_set_chunk_pages(int(pages)))


def decode_set_merge_in_place(max_chunks: int):
    """Merge split sequences inside the decode kernel when they have at most max_chunks chunks
    (0: always the separate combine kernel)."""
    _check(lib().pkv_decode_set_merge_in_place(int(max_chunks)))


def decode_set_kernel(which: int):
    """0 automatic, 1 CUDA-core decode kernel, 2 tensor-core decode kernel."""
    _check(lib().pkv_decode_set_kernel(int(which)))


def decode_set_split(mode: int):
    """0 automatic (the split autotuning recorded for the call's shape, else chunks), 1 chunks
    only, 2 the balanced split of the tensor-core decode wherever it applies, 3 and 4 chunks
    1.5 and 2 times the automatic length wherever they apply."""
    _check(lib().pkv_decode_set_split(int(mode)))


def decode_set_autotune(on: bool):
    """Time every split that applies on the first call of each shape and keep the fastest
    (pkv.h)."""
    _check(lib().pkv_decode_set_autotune(1 if on else 0))


def decode_autotune_reset():
    _check(lib().pkv_decode_autotune_reset())


def decode_split_choice(kv_dtype, q_dtype, batch, num_q_heads, num_kv_heads, max_pages_per_seq,
                        window=0, sink_tokens=0, fused=False) -> int:
    """The recorded split for a shape: 0 chunks, 1 balanced, 2 and 3 chunks 1.5 and 2 times
    longer, -1 none. Dtypes as torch dtypes or pkv_dtype codes."""
    code = lambda d: d if isinstance(d, int) else _dtype_code(torch.empty(0, dtype=d))
    return int(lib().pkv_decode_split_choice(code(kv_dtype), code(q_dtype), batch, num_q_heads,
                                             num_kv_heads, max_pages_per_seq, window, sink_tokens,
                                             1 if fused else 0))


def decode_chunk_pages(batch, num_kv_heads, max_pages_per_seq) -> int:
    return int(lib().pkv_decode_chunk_pages(batch, num_kv_heads, max_pages_per_seq))


def pages_needed(n_tokens: int, page_size: int = 16) -> int:
    out = ctypes.c_int64(0)
    _check(lib().pkv_pages_needed(int(n_tokens), int(page_size), ctypes.byref(out)))
    return int(out.value)


def slot_mapping(block_tables, positions, num_pages, requests=None, page_size=16) -> np.ndarray:
    """Host slot mapping: int64 slots of (request, position) pairs through host page tables."""
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    req = None if requests is None else np.ascontiguousarray(np.asarray(requests, dtype=np.int32))
    out = np.empty(len(pos), dtype=np.int64)
    _check(lib().pkv_slot_mapping(bt.ctypes.data, bt.shape[1],
                                  None if req is None else req.ctypes.data, pos.ctypes.data,
                                  len(pos), page_size, int(num_pages), out.ctypes.data))
    return out


class PageAllocator:
    """Host page allocator: O(1) LIFO free list with reference counts (pkv_allocator_*)."""

    def __init__(self, num_pages: int, initial_free_order=None):
        self._h = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(np.asarray(initial_free_order, dtype=np.int32))
        _check(lib().pkv_allocator_create(int(num_pages),
                                          None if order is None else order.ctypes.data,
                                          ctypes.byref(self._h)))
        self.num_pages = int(num_pages)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_allocator_destroy(h)
            self._h = None

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(max(n, 0), dtype=np.int32)
        _check(lib().pkv_alloc(self._h, int(n), out.ctypes.data if n > 0 else None))
        return out

    def incref(self, ids):
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        _check(lib().pkv_incref(self._h, a.ctypes.data if a.size else None, a.size))

    def decref(self, ids):
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        _check(lib().pkv_decref(self._h, a.ctypes.data if a.size else None, a.size))

    def num_free(self) -> int:
        return int(lib().pkv_num_free(self._h))

    def refcount(self, page_id: int) -> int:
        return int(lib().pkv_refcount(self._h, int(page_id)))

    def cow_page(self, row: list, position: int, page_size: int = 16):
        """Copy-on-write for a write at ``position`` of a request with pages ``row`` (updated
        in place). Returns (src, dst) to copy, or None when the page is private."""
        r = (ctypes.c_int32 * max(len(row), 1))(*[int(x) for x in row])
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        _check(lib().pkv_cow_page(self._h, r, len(row), int(position), int(page_size),
                                  ctypes.byref(src), ctypes.byref(dst)))
        row[:] = list(r)[:len(row)]
        return None if src.value < 0 else (int(src.value), int(dst.value))


def _ids(rids) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(rids if isinstance(rids, np.ndarray) else list(rids),
                                           dtype=np.int64))


def _counts(counts) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(counts if isinstance(counts, np.ndarray)
                                           else list(counts), dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data if a.size else None


def _host_int32(a, shape, name):
    """``a`` if it is a C-contiguous int32 host array (numpy, or a CPU tensor) of ``shape``;
    the library writes through its address."""
    if isinstance(a, torch.Tensor):
        ok = (a.device.type == "cpu" and a.dtype == torch.int32 and a.is_contiguous() and
              tuple(a.shape) == tuple(shape))
    else:
        ok = (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous and
              a.flags.writeable and a.shape == tuple(shape))
    if not ok:
        raise PkvError(-2, "%s must be a C-contiguous int32 host array of shape %s" %
                       (name, tuple(shape)))
    return a


class SeqTable:
    """Request page tables over a PageAllocator (pkv_seq_*): rows of page ids and token counts,
    fork / free / reserve (with copy-on-write) / window release, all in the C library."""

    def __init__(self, allocator: PageAllocator, page_size: int = 16):
        self._alloc = allocator  # the allocator outlives the table
        self._h = ctypes.c_void_p()
        _check(lib().pkv_seq_table_create(allocator._h, int(page_size), ctypes.byref(self._h)))
        self.page_size = int(page_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_seq_table_destroy(h)
            self._h = None

    def add(self, rid: int, shared_pages=None, shared_len: int = 0, adopt: bool = False):
        """A new request, optionally on whole shared pages; ``adopt``: the request takes over
        references the caller holds on them instead of taking new ones."""
        fn = lib().pkv_seq_adopt if adopt else lib().pkv_seq_add
        if shared_pages is None:
            _check(fn(self._h, int(rid), None, 0, int(shared_len)))
            return
        p = np.ascontiguousarray(np.asarray(list(shared_pages), dtype=np.int32))
        _check(fn(self._h, int(rid), _ptr(p), p.size, int(shared_len)))

    def fork(self, src_rids, new_rids):
        s, n = _ids(src_rids), _ids(new_rids)
        if s.size != n.size:
            raise PkvError(-1, "src_rids and new_rids differ in length")
        _check(lib().pkv_seq_fork(self._h, _ptr(s), _ptr(n), s.size))

    def free(self, rids):
        r = _ids(rids)
        _check(lib().pkv_seq_free(self._h, _ptr(r), r.size))

    def reserve(self, rids, counts):
        """Returns (int64 slots of the new positions, list of (src, dst) pages to copy)."""
        r, c = _ids(rids), _counts(counts)
        if r.size != c.size:
            raise PkvError(-1, "rids and counts differ in length")
        slots = np.empty(int(c.sum()) if c.size else 0, dtype=np.int64)
        src = np.empty(max(r.size, 1), dtype=np.int32)
        dst = np.empty_like(src)
        nc = ctypes.c_int32(0)
        _check(lib().pkv_seq_reserve(self._h, _ptr(r), _ptr(c), r.size, _ptr(slots),
                                     src.ctypes.data, dst.ctypes.data, ctypes.byref(nc)))
        return slots, [(int(src[i]), int(dst[i])) for i in range(nc.value)]

    def tables(self, rids, width: int | None = None, out=None):
        """Block-table rows int32 [n][width] of the requests (unused columns 0, released pages
        -1); ``out`` (a contiguous int32 numpy array or CPU tensor) is filled in place."""
        r = _ids(rids)
        if width is None:
            width = max([self.num_pages_of(x) for x in r.tolist()] + [1])
        bt = np.empty((r.size, int(width)), dtype=np.int32) if out is None else out
        bt_p = bt.data_ptr() if isinstance(bt, torch.Tensor) else bt.ctypes.data
        _check(lib().pkv_seq_tables(self._h, _ptr(r), r.size, int(width),
                                    bt_p if r.size else None, None))
        return bt

    def lengths(self, rids, out=None):
        """Token counts (int32 [n]) of the requests; ``out`` is filled in place when given."""
        r = _ids(rids)
        cl = np.empty(r.size, dtype=np.int32) if out is None else out
        cl_p = cl.data_ptr() if isinstance(cl, torch.Tensor) else cl.ctypes.data
        _check(lib().pkv_seq_tables(self._h, _ptr(r), r.size, 0, None, cl_p if r.size else None))
        return cl

    def step(self, free_rids, new_rids, prompt_counts, live_rids, width=None, tables_out=None,
             lens_out=None, live_slots=False, incremental=False):
        """One scheduler step (pkv_seq_step): drop ``free_rids``, add ``new_rids`` grown by their
        ``prompt_counts``, grow every one of ``live_rids`` by one token and export their table
        rows (``width`` columns; into ``tables_out`` when given, else a new array) and lengths
        (into ``lens_out``). ``incremental``: rows still holding the same request from the
        previous incremental step into the same ``tables_out`` are only patched (the caller
        leaves them alone in between). Returns (prompt slots int64, tables, lengths, copy
        pairs), plus the live requests' new slots when ``live_slots``."""
        f, nw, c, lv = _ids(free_rids), _ids(new_rids), _counts(prompt_counts), _ids(live_rids)
        if nw.size != c.size:
            raise PkvError(-1, "new_rids and prompt_counts differ in length")
        n = lv.size
        if width is None:
            w = ctypes.c_int32(0)
            _check(lib().pkv_seq_step_width(self._h, _ptr(nw), _ptr(c), nw.size, _ptr(lv), n,
                                            ctypes.byref(w)))
            width = w.value
        if tables_out is None:
            # a fresh array every call: the previous call's rows are not in it
            incremental = False
            bt = np.empty((n, int(width)), dtype=np.int32)
        else:
            bt = _host_int32(tables_out, (n, int(width)), "tables_out")
        cl = np.empty(n, dtype=np.int32) if lens_out is None else _host_int32(lens_out, (n,),
                                                                              "lens_out")
        ptr = (lambda a: a.data_ptr() if isinstance(a, torch.Tensor) else a.ctypes.data)
        ps = np.empty(int(c.sum()) if c.size else 0, dtype=np.int64)
        ls = np.empty(n, dtype=np.int64) if live_slots else None
        src = np.empty(max(n, 1), dtype=np.int32)
        dst = np.empty_like(src)
        nc = ctypes.c_int32(0)
        _check(lib().pkv_seq_step(self._h, _ptr(f), f.size, _ptr(nw), _ptr(c), nw.size, _ptr(ps),
                                  _ptr(lv), n, None if ls is None else _ptr(ls), int(width),
                                  ptr(bt) if n else None, ptr(cl) if n else None,
                                  int(bool(incremental)), src.ctypes.data, dst.ctypes.data,
                                  ctypes.byref(nc)))
        copies = [(int(src[i]), int(dst[i])) for i in range(nc.value)]
        return (ps, bt, cl, copies) + ((ls,) if live_slots else ())

    def release_outside_window(self, rid: int, window: int, sink_tokens: int = 0) -> int:
        n = ctypes.c_int32(0)
        _check(lib().pkv_seq_release_outside_window(self._h, int(rid), int(window),
                                                    int(sink_tokens), ctypes.byref(n)))
        return int(n.value)

    def length(self, rid: int) -> int:
        n = int(lib().pkv_seq_len(self._h, int(rid)))
        if n < 0:
            raise KeyError(rid)
        return n

    def num_pages_of(self, rid: int) -> int:
        n = int(lib().pkv_seq_pages(self._h, int(rid), None, 0))
        if n < 0:
            raise KeyError(rid)
        return n

    def pages(self, rid: int) -> list:
        n = self.num_pages_of(rid)
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().pkv_seq_pages(self._h, int(rid), out.ctypes.data, n)
        return [int(x) for x in out[:n]]

    def ids(self) -> list:
        n = int(lib().pkv_seq_count(self._h))
        out = np.empty(max(n, 1), dtype=np.int64)
        m = int(lib().pkv_seq_ids(self._h, out.ctypes.data, n))
        return [int(x) for x in out[:min(n, m)]]


class PrefixCache:
    """Prompt-prefix page cache over a PageAllocator (pkv_prefix_*): whole pages, keyed by
    tenant and tokens, exact matches only."""

    def __init__(self, allocator: PageAllocator, page_size: int = 16):
        self._alloc = allocator  # keeps the allocator alive while the cache exists
        self._h = ctypes.c_void_p()
        _check(lib().pkv_prefix_cache_create(allocator._h, int(page_size), ctypes.byref(self._h)))
        self.page_size = page_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_prefix_cache_destroy(h)
            self._h = None

    def lookup(self, tenant: int, tokens, max_pages: int = 1 << 20) -> list:
        """Pages of the longest cached prefix (the caller gets a reference on each)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        cap = min(max_pages, t.size)  # room for any whole-page count; the library counts them
        out = np.empty(max(cap, 1), dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(lib().pkv_prefix_lookup(self._h, int(tenant), t.ctypes.data if t.size else None,
                                       t.size, out.ctypes.data, cap, ctypes.byref(n)))
        return [int(x) for x in out[:n.value]]

    def insert(self, tenant: int, tokens, pages):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        p = np.ascontiguousarray(np.asarray(pages, dtype=np.int32))
        _check(lib().pkv_prefix_insert(self._h, int(tenant), t.ctypes.data if t.size else None,
                                       t.size, p.ctypes.data if p.size else None, p.size))

    def evict(self, max_pages: int) -> int:
        n = ctypes.c_int32(0)
        _check(lib().pkv_prefix_evict(self._h, int(max_pages), ctypes.byref(n)))
        return int(n.value)

    def size(self) -> int:
        return int(lib().pkv_prefix_size(self._h))

    def insert_request(self, tenant: int, tokens, table: SeqTable, rid: int):
        """Caches the full pages of request ``rid``'s prompt ``tokens`` (already written)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        _check(lib().pkv_prefix_insert_request(self._h, int(tenant), _ptr(t), t.size, table._h,
                                               int(rid)))

    def add_request(self, table: SeqTable, rid: int, tenant: int, tokens) -> int:
        """New request ``rid`` in ``table`` starting on the longest cached prefix of its prompt
        ``tokens`` (the lookup's references become the request's); returns the prompt tokens
        already cached."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = ctypes.c_int64(0)
        _check(lib().pkv_seq_add_cached_prefix(table._h, int(rid), self._h, int(tenant), _ptr(t),
                                               t.size, ctypes.byref(n)))
        return int(n.value)


def trace_enable(on: bool = True):
    _check(lib().pkv_trace_enable(1 if on else 0))


def trace_reset():
    _check(lib().pkv_trace_reset())


def trace_read(kernel: str):
    """(launches, total device ms) for a kernel family since the last reset."""
    n = ctypes.c_int32(0)
    ms = ctypes.c_double(0.0)
    _check(lib().pkv_trace_read(kernel.encode(), ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)
