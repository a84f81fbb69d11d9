"""CPU oracle for paged decode attention and its host logic -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
(``bench.py``'s ``cpu_baseline`` and ``--impl reference``) may import this package. The CUDA
library never calls it, and it never calls the CUDA library: the two share no code.

Everything here is the plain definition the KV-cache pages give, written in fp64 (attention,
in ``pkv_oracle.c``) or in integer numpy / Python (page accounting, slot mapping, the
append scatter, the page allocator model):

* ``kv_bytes_per_token`` / ``total_kv_bytes`` -- "KV cache and PagedAttention", section 2
  (Memory cost): per token 2 * L * h_kv * d_h * b; for batch B and length T,
  2 * B * T * L * d_kv * b with d_kv = h_kv * d_h.
* ``pages_needed`` / ``wasted_slots`` -- section 4 (PagedAttention): fixed 16-token pages; a
  17-token request takes 2 pages and leaves 15 slots unused.
* ``slot_of`` / ``slot_mapping`` / ``scatter_append`` / ``gather_contiguous`` -- section 4:
  a per-request page table lists page indices in a pool; token position p of a request lives
  in page ``table[p // P]`` at row ``p % P`` (reading: the pages never write this formula
  out; it is the only one consistent with "page table: list of page indices" and fixed-size
  pages). The write phase ("KV Cache" glossary, write/read phase) appends the new token's
  K and V there.
* ``AllocatorModel`` -- section 4: uniform pages, O(1) allocator; pages shared between
  requests ("Sharing", and the glossary's "Blocks can be shared across sequences") are
  reference-counted (reading: the counting scheme is not on the pages). Free list is LIFO.
* ``decode_*`` -- section 1 (The setup) and the "Memoizing Context" page: softmax attention
  of the new token's query over all cached keys and values. GQA grouping reading: query head
  h uses KV head h // (h_q // h_kv). Section 8 (sliding-window cache and attention sinks):
  with a window of W tokens only the last W are attended, plus the first S "sink" tokens when
  S > 0 (reading: the pages give W and S as counts of positions; W = 0 means no window).
* ``e4m3_*`` / ``quantize_e4m3`` / ``absmax_scale`` -- section 7 (KV cache quantisation,
  "fp8 KV (E4M3)"): code values per the OCP FP8 E4M3 format; readings: per-(layer, kv head)
  scale s = fp32(absmax / 448) (1 when absmax is 0), code = RNE-with-saturation of
  fp32(x / s).
* ``quantize_int8`` -- section 7, "INT8 KV: similar" (no scheme given); reading: symmetric
  codes in [-127, 127], s = fp32(absmax / 127), code = fp32(x / s) rounded half-to-even and
  clamped.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

F32, BF16, E4M3, INT8 = 0, 1, 2, 3
_DT = {"f32": F32, "bf16": BF16, "fp8_e4m3": E4M3, "int8": INT8}

_lib = None


def bind(L):
    """Declare the C oracle's entry points on a loaded library ``L`` and return it."""
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    L.oracle_e4m3_value.restype = ctypes.c_double
    L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_quantize_e4m3.restype = None
    L.oracle_quantize_e4m3.argtypes = [vp, i64, ctypes.c_float, vp]
    L.oracle_quantize_int8.restype = None
    L.oracle_quantize_int8.argtypes = [vp, i64, ctypes.c_float, vp]
    L.oracle_attend.restype = None
    L.oracle_attend.argtypes = [vp, vp, vp, i64, i32, dbl, vp]
    L.oracle_paged_decode.restype = i32
    L.oracle_paged_decode.argtypes = [vp, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32,
                                      vp, i32, vp, dbl, vp, vp, vp, i32, vp, i32, i32, i32]
    L.oracle_contiguous_decode.restype = i32
    L.oracle_contiguous_decode.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, i32, i32,
                                           i32, vp, vp, dbl, vp, vp, vp, i32, vp, i32, i32,
                                           i32]
    L.oracle_max_threads.restype = i32
    L.oracle_max_threads.argtypes = []
    return L


def lib():
    """The compiled C oracle (built on first use)."""
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(_build.build()))
    return _lib


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ---- memory formula and page accounting (integers) -----------------------------------------

def kv_bytes_per_token(L: int, h_kv: int, d_h: int, b: int) -> int:
    """2 * L * h_kv * d_h * b bytes: one K and one V vector per layer and KV head."""
    return 2 * L * h_kv * d_h * b


def total_kv_bytes(B: int, T: int, L: int, d_kv: int, b: int) -> int:
    """2 * B * T * L * d_kv * b bytes for batch B at sequence length T."""
    return 2 * B * T * L * d_kv * b


def pages_needed(n_tokens: int, page_size: int = 16) -> int:
    """Fixed-size pages a request of n tokens occupies: the smallest count holding n."""
    pages = 0
    while pages * page_size < n_tokens:
        pages += 1
    return pages


def wasted_slots(n_tokens: int, page_size: int = 16) -> int:
    return pages_needed(n_tokens, page_size) * page_size - n_tokens


def slot_of(table_row, position: int, page_size: int = 16) -> int:
    """Physical slot of a logical token position: page table[p // P], row p % P."""
    return int(table_row[position // page_size]) * page_size + position % page_size


def slot_mapping(block_tables: np.ndarray, positions: np.ndarray, page_size: int = 16,
                 requests: np.ndarray | None = None) -> np.ndarray:
    """int64 slots for tokens at ``positions`` of ``requests`` (default: token i of request i);
    a negative position maps to -1 (padding, skipped by the append)."""
    positions = np.asarray(positions)
    if requests is None:
        requests = np.arange(len(positions))
    out = np.empty(len(positions), dtype=np.int64)
    for i, (b, p) in enumerate(zip(requests, positions)):
        out[i] = -1 if p < 0 else slot_of(block_tables[b], int(p), page_size)
    return out


def scatter_append(pool: np.ndarray, slots: np.ndarray, new: np.ndarray, page_size: int = 16):
    """Write phase: pool[slot // P, :, slot % P, :] = new[i] for every slot >= 0.

    pool is [num_pages, h_kv, P, d] (any element type), new is [N, h_kv, d]."""
    for i, s in enumerate(np.asarray(slots)):
        if s < 0:
            continue
        pool[s // page_size, :, s % page_size, :] = new[i]
    return pool


def gather_contiguous(pool: np.ndarray, table_row, n_tokens: int, page_size: int = 16):
    """Read phase through the page table: the request's [n_tokens, h_kv, d] in logical order."""
    rows = [pool[table_row[t // page_size], :, t % page_size, :] for t in range(n_tokens)]
    if not rows:
        return pool[:0, :, 0, :]
    return np.stack(rows, 0)


class AllocatorModel:
    """Page allocator model: LIFO free list, reference counts, all-or-nothing requests.

    ``initial_order`` lists the free pages; the first entry is handed out first."""

    def __init__(self, num_pages: int, initial_order=None):
        order = list(range(num_pages)) if initial_order is None else [int(x) for x in initial_order]
        self.num_pages = num_pages
        self.free = list(reversed(order))  # top of the stack = end of the list
        self.ref = [0] * num_pages

    def alloc(self, n: int):
        if n < 0:
            raise ValueError("negative count")
        if n > len(self.free):
            raise MemoryError("out of pages")
        ids = [self.free.pop() for _ in range(n)]
        for i in ids:
            self.ref[i] = 1
        return ids

    def _check(self, ids, need):
        counts = {}
        for i in ids:
            if not 0 <= i < self.num_pages:
                raise IndexError("page id out of range")
            counts[i] = counts.get(i, 0) + 1
        for i, c in counts.items():
            if self.ref[i] < need(c):
                raise ValueError("reference count")

    def incref(self, ids):
        self._check(ids, lambda c: 1)
        for i in ids:
            self.ref[i] += 1

    def decref(self, ids):
        self._check(ids, lambda c: c)
        for i in ids:
            self.ref[i] -= 1
            if self.ref[i] == 0:
                self.free.append(i)

    def num_free(self) -> int:
        return len(self.free)


class PrefixCacheModel:
    """Prompt-prefix page cache model ("KV cache and PagedAttention", section 6; tenant in the
    key per pitfall 5): entry i of a prompt is the exact (tenant, tokens of pages 0..i); a
    lookup returns the pages of the longest cached prefix in whole pages and references them;
    the cache holds one reference per entry; eviction removes, in passes over least-recently-
    used order, entries with no cached continuation whose page only the cache references."""

    def __init__(self, allocator: AllocatorModel, page_size: int = 16):
        self.a = allocator
        self.P = page_size
        self.entries = {}  # key -> page
        self.lru = []  # keys, least recently used first

    def _touch(self, key):
        self.lru.remove(key)
        self.lru.append(key)

    def _key(self, tenant, tokens, i):
        return (tenant, tuple(int(t) for t in tokens[:(i + 1) * self.P]))

    def lookup(self, tenant, tokens, max_pages=1 << 20):
        hits = []
        for i in range(min(len(tokens) // self.P, max_pages)):
            key = self._key(tenant, tokens, i)
            if key not in self.entries:
                break
            hits.append(key)
        pages = [self.entries[k] for k in hits]
        if pages:
            self.a.incref(pages)
        for k in hits:
            self._touch(k)
        return pages

    def insert(self, tenant, tokens, pages):
        for i in range(min(len(tokens) // self.P, len(pages))):
            key = self._key(tenant, tokens, i)
            if key in self.entries:
                self._touch(key)
                continue
            self.a.incref([pages[i]])
            self.entries[key] = pages[i]
            self.lru.append(key)

    def _children(self, key):
        return sum(1 for k in self.entries
                   if k[0] == key[0] and len(k[1]) == len(key[1]) + self.P and k[1][:len(key[1])] == key[1])

    def evict(self, max_pages):
        done, progress = 0, True
        while done < max_pages and progress:
            progress = False
            for key in list(self.lru):
                if done >= max_pages:
                    break
                if key not in self.entries:
                    continue
                page = self.entries[key]
                if self._children(key) == 0 and self.a.ref[page] == 1:
                    self.a.decref([page])
                    del self.entries[key]
                    self.lru.remove(key)
                    done += 1
                    progress = True
        return done


# ---- FP8 E4M3 -------------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y: float) -> int:
    return int(lib().oracle_e4m3_encode(float(y)))


def quantize_e4m3(x: np.ndarray, s: float) -> np.ndarray:
    """uint8 codes of fp32(x / s); x is converted to float32 first (exact for bf16 input)."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(xf.shape, dtype=np.uint8)
    lib().oracle_quantize_e4m3(xf.ctypes.data, xf.size, ctypes.c_float(s), out.ctypes.data)
    return out


def absmax_scale(x: np.ndarray, qmax: float = 448.0) -> np.float32:
    """fp32(max |x| / qmax), or 1 when every element is zero. x: float32 values; qmax 448 for
    E4M3 codes, 127 for INT8 codes."""
    a = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else np.float32(0)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a) / np.float32(qmax)


def absmax_scales_per_head(x: np.ndarray, qmax: float = 448.0) -> np.ndarray:
    """x: [tokens, h_kv, d] float32 -> float32 [h_kv] scales, one per KV head."""
    return np.array([absmax_scale(x[:, j, :], qmax) for j in range(x.shape[1])],
                    dtype=np.float32)


def quantize_int8(x: np.ndarray, s: float) -> np.ndarray:
    """int8 codes: fp32(x / s) rounded to nearest (ties to even), clamped to [-127, 127]."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(xf.shape, dtype=np.int8)
    lib().oracle_quantize_int8(xf.ctypes.data, xf.size, ctypes.c_float(s), out.ctypes.data)
    return out


# ---- conversions of torch CPU tensors to what the C oracle reads ---------------------------

def as_raw(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Contiguous numpy view holding the exact stored bits of a CPU tensor."""
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp8_e4m3":
        if t.dtype == torch.uint8:
            return t.numpy()
        return t.view(torch.uint8).numpy()
    if dtype == "int8":
        return t.view(torch.int8).numpy()
    return t.to(torch.float32).numpy()


def _ptr(a):
    return None if a is None else a.ctypes.data


def _pairs_arg(pairs):
    if pairs is None:
        return None, 0
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return p, len(p)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One query [d] over K, V [T, d] (float64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.zeros(q.shape[0], dtype=np.float64)
    lib().oracle_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], q.shape[0],
                        float(scale), out.ctypes.data)
    return out


def paged_decode(q_raw, q_dtype, k_pool_raw, v_pool_raw, kv_dtype, block_tables, context_lens,
                 scale, k_scales=None, v_scales=None, pairs=None, n_threads=0, sink=0, window=0):
    """Decode attention through page tables. Pools: [num_pages, h_kv, P, d] raw arrays.
    window > 0 keeps only the last ``window`` tokens plus the first ``sink`` ones.

    Returns float64 [B, h_q, d], or [n_pairs, d] when ``pairs`` ((b, h) rows) is given."""
    q_raw = np.ascontiguousarray(q_raw)
    B, h_q, d = q_raw.shape
    num_pages, h_kv, P, d2 = k_pool_raw.shape
    assert d2 == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ks = None if k_scales is None else np.ascontiguousarray(k_scales, dtype=np.float32)
    vs = None if v_scales is None else np.ascontiguousarray(v_scales, dtype=np.float32)
    p, n = _pairs_arg(pairs)
    out = np.zeros((n, d) if p is not None else (B, h_q, d), dtype=np.float64)
    kp = np.ascontiguousarray(k_pool_raw)
    vp = np.ascontiguousarray(v_pool_raw)
    st = lib().oracle_paged_decode(q_raw.ctypes.data, _DT[q_dtype], B, h_q, d, kp.ctypes.data,
                                   vp.ctypes.data, _DT[kv_dtype], num_pages, h_kv, P,
                                   bt.ctypes.data, bt.shape[1], cl.ctypes.data, float(scale),
                                   _ptr(ks), _ptr(vs), _ptr(p), n, out.ctypes.data, n_threads,
                                   int(sink), int(window))
    if st != 0:
        raise IndexError("page id out of range in a block table")
    return out


def contiguous_decode(q_raw, q_dtype, k_rows_raw, v_rows_raw, kv_dtype, offsets, context_lens,
                      scale, k_scales=None, v_scales=None, prefix_k_raw=None, prefix_v_raw=None,
                      prefix_len=0, pairs=None, n_threads=0, sink=0, window=0):
    """Decode attention over contiguous per-request rows (the naive cache).

    k_rows_raw: [rows, h_kv, d]; request b's own tokens start at row offsets[b]; with a
    shared prefix the first prefix_len tokens come from prefix_*_raw [prefix_len, h_kv, d]."""
    q_raw = np.ascontiguousarray(q_raw)
    B, h_q, d = q_raw.shape
    h_kv = k_rows_raw.shape[1]
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ks = None if k_scales is None else np.ascontiguousarray(k_scales, dtype=np.float32)
    vs = None if v_scales is None else np.ascontiguousarray(v_scales, dtype=np.float32)
    p, n = _pairs_arg(pairs)
    out = np.zeros((n, d) if p is not None else (B, h_q, d), dtype=np.float64)
    kr = np.ascontiguousarray(k_rows_raw)
    vr = np.ascontiguousarray(v_rows_raw)
    pk = None if prefix_k_raw is None else np.ascontiguousarray(prefix_k_raw)
    pv = None if prefix_v_raw is None else np.ascontiguousarray(prefix_v_raw)
    lib().oracle_contiguous_decode(q_raw.ctypes.data, _DT[q_dtype], B, h_q, d, kr.ctypes.data,
                                   vr.ctypes.data, _ptr(pk), _ptr(pv), int(prefix_len),
                                   _DT[kv_dtype], h_kv, off.ctypes.data, cl.ctypes.data,
                                   float(scale), _ptr(ks), _ptr(vs), _ptr(p), n,
                                   out.ctypes.data, n_threads, int(sink), int(window))
    return out


def attended_tokens(T: int, sink: int = 0, window: int = 0):
    """Token positions a request of T tokens attends: all when window is 0, else the last
    ``window`` plus the first ``sink`` ("KV cache and PagedAttention", section 8)."""
    if window <= 0:
        return list(range(T))
    return [t for t in range(T) if t >= T - window or t < sink]


def decode_inputs(w, pairs=None, n_threads=0, k_scales=None, v_scales=None, k_codes=None,
                  v_codes=None, sink=0, window=0):
    """Expected decode output for a ``workloads.DecodeInputs`` from its contiguous tokens.

    For an FP8 cache pass the per-head scales and the codes (uint8, same layout as
    ``w.k_tokens``) the oracle's own quantiser produced."""
    qd = w.q_dtype
    q_raw = as_raw(w.q, qd)
    if w.kv_dtype in ("fp8_e4m3", "int8"):
        kr, vr, kvd = k_codes, v_codes, w.kv_dtype
        pk = pv = None
        if w.prefix_len:
            raise NotImplementedError("quantised cache with a shared prefix")
    else:
        kvd = w.kv_dtype
        kr, vr = as_raw(w.k_tokens, kvd), as_raw(w.v_tokens, kvd)
        pk = as_raw(w.prefix_k, kvd) if w.prefix_len else None
        pv = as_raw(w.prefix_v, kvd) if w.prefix_len else None
    return contiguous_decode(q_raw, qd, kr, vr, kvd, w.offsets, w.context_lens, w.scale,
                             k_scales, v_scales, pk, pv, w.prefix_len, pairs, n_threads, sink,
                             window)
