"""ctypes binding of the libv4a page allocator (v4a_pages.h): argument
marshalling only; the planning and the free lists are the library's C++.

Source: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Method
details, "keeping the KV cache memory packed" (one logical block of 256
native positions in every layer, compressor state kept as sliding-window
state in the same pools, page sizes folded into a few buckets with one pool
each).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import v4a

BLOCK, RING = 0, 1
ERR_OUT_OF_PAGES = 6


class Kind(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layers", C.c_int32), ("page_bytes", C.c_int64),
                ("slot_bytes", C.c_int64), ("ring_slots", C.c_int32), ("bucket", C.c_int32)]


class KindInfo(C.Structure):
    _fields_ = [("bucket", C.c_int32), ("slots", C.c_int32), ("ring_pages", C.c_int32),
                ("ring_cap", C.c_int32), ("table_cols", C.c_int32), ("table_offset", C.c_int64),
                ("table_stride", C.c_int64)]


_sigs_done = False


def _lib() -> C.CDLL:
    global _sigs_done
    L = v4a.lib()
    if not _sigs_done:
        P = C.c_void_p
        L.v4a_pages_create.argtypes = [C.POINTER(Kind), C.c_int32, C.c_int32, C.c_int32, C.c_int64,
                                       C.POINTER(P)]
        L.v4a_pages_destroy.argtypes = [P]
        L.v4a_pages_destroy.restype = None
        L.v4a_pages_num_buckets.argtypes = [P]
        L.v4a_pages_bucket.argtypes = [P, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                       C.POINTER(C.c_int64)]
        L.v4a_pages_info.argtypes = [P, C.c_int32, C.POINTER(KindInfo)]
        L.v4a_pages_tables.argtypes = [P, C.POINTER(C.c_int64)]
        L.v4a_pages_tables.restype = C.POINTER(C.c_int32)
        L.v4a_pages_open.argtypes = [P, C.c_int32]
        L.v4a_pages_reserve.argtypes = [P, C.c_int32, C.c_int64]
        L.v4a_pages_close.argtypes = [P, C.c_int32]
        L.v4a_pages_blocks.argtypes = [P, C.c_int32]
        L.v4a_pages_blocks.restype = C.c_int64
        _sigs_done = True
    return L


def block_kind(page_bytes: int, layers: int) -> Kind:
    """A compressed cache: one page of `page_bytes` per 256-position block per layer."""
    return Kind(BLOCK, layers, page_bytes, 0, 0, 0)


def ring_kind(slot_bytes: int, ring_slots: int, bucket: int, layers: int) -> Kind:
    """A sliding-window ring of at least `ring_slots` slots in bucket rank `bucket`."""
    return Kind(RING, layers, 0, slot_bytes, ring_slots, bucket)


@dataclass
class Bucket:
    page_bytes: int
    num_pages: int
    free_pages: int


class PageAllocator:
    """Owns a v4a_pages handle; the tables are a numpy view of the library's
    host array (valid while the allocator lives)."""

    def __init__(self, kinds: list, max_seqs: int, max_blocks: int, budget_bytes: int):
        self._L = _lib()
        arr = (Kind * len(kinds))(*kinds)
        h = C.c_void_p()
        rc = self._L.v4a_pages_create(arr, len(kinds), max_seqs, max_blocks, budget_bytes, C.byref(h))
        v4a._check("v4a_pages_create", rc)
        self._h = h
        self.num_kinds = len(kinds)
        self.max_seqs, self.max_blocks = max_seqs, max_blocks

    def close_handle(self):
        if getattr(self, "_h", None):
            self._L.v4a_pages_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close_handle()

    # ---- plan ----------------------------------------------------------------
    @property
    def num_buckets(self) -> int:
        return self._L.v4a_pages_num_buckets(self._h)

    def bucket(self, b: int) -> Bucket:
        pb, n, f = C.c_int64(), C.c_int64(), C.c_int64()
        v4a._check("v4a_pages_bucket", self._L.v4a_pages_bucket(self._h, b, C.byref(pb), C.byref(n), C.byref(f)))
        return Bucket(pb.value, n.value, f.value)

    def buckets(self) -> list:
        return [self.bucket(b) for b in range(self.num_buckets)]

    def info(self, kind: int) -> KindInfo:
        i = KindInfo()
        v4a._check("v4a_pages_info", self._L.v4a_pages_info(self._h, kind, C.byref(i)))
        return i

    def tables(self) -> np.ndarray:
        """Every table as one int32 array (a view, not a copy)."""
        n = C.c_int64()
        ptr = self._L.v4a_pages_tables(self._h, C.byref(n))
        return np.ctypeslib.as_array(ptr, shape=(n.value,))

    def table(self, kind: int, layer: int) -> np.ndarray:
        """The [max_seqs][table_cols] table of one kind and layer (a view)."""
        i = self.info(kind)
        t = self.tables()
        off = i.table_offset + layer * i.table_stride
        return t[off: off + i.table_stride].reshape(self.max_seqs, i.table_cols)

    # ---- sequences -------------------------------------------------------------
    def open(self, seq: int):
        v4a._check("v4a_pages_open", self._L.v4a_pages_open(self._h, seq))

    def reserve(self, seq: int, positions: int):
        v4a._check("v4a_pages_reserve", self._L.v4a_pages_reserve(self._h, seq, positions))

    def close(self, seq: int):
        v4a._check("v4a_pages_close", self._L.v4a_pages_close(self._h, seq))

    def blocks(self, seq: int) -> int:
        return int(self._L.v4a_pages_blocks(self._h, seq))
