"""ctypes binding of libv4a (argument marshalling only).

Every function here builds the C argument structs from torch CUDA tensors and
calls the library; all arithmetic runs in the CUDA kernels.  If libv4a.so is
missing the first call raises: there is no CPU or eager fallback.
"""
from __future__ import annotations

import ctypes as C
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libv4a.so")

V4A_OK = 0
ERRORS = {1: "invalid argument", 2: "unsupported", 3: "ring too small", 4: "workspace", 5: "cuda",
          6: "out of pages"}
DEV_BAD_BLOCK, DEV_BAD_BATCH, DEV_BAD_INDEX = 1, 2, 4
KV_BF16, KV_FP8_TOKEN = 0, 1
IX_BF16, IX_FP8_B128, IX_FP4_B32, IX_FP4_MX32 = 0, 1, 2, 3
Q_BF16, Q_FP8_HEAD = 0, 1
OUT_BF16, OUT_FP8_TOKEN = 0, 1

_p = C.c_void_p


class Batch(C.Structure):
    _fields_ = [("num_tokens", C.c_int32), ("seq_ids", _p), ("positions", _p),
                ("num_seqs", C.c_int32), ("max_new_per_seq", C.c_int32)]


class Cache(C.Structure):
    _fields_ = [("ratio", C.c_int32), ("dim", C.c_int32), ("rope_dims", C.c_int32),
                ("rope_theta", C.c_float), ("format", C.c_int32), ("pool", _p),
                ("num_blocks", C.c_int64), ("block_table", _p), ("max_blocks", C.c_int32)]


class RingPages(C.Structure):
    _fields_ = [("pool", _p), ("num_pages", C.c_int64), ("page_bytes", C.c_int64), ("table", _p),
                ("slots", C.c_int32)]


class Compressor(C.Structure):
    _fields_ = [("cache", Cache), ("x", _p), ("gate", _p), ("bias", _p), ("gamma", _p),
                ("eps", C.c_float), ("ring_x", _p), ("ring_gate", _p), ("ring_cap", C.c_int32),
                ("ring_pages", C.POINTER(RingPages))]


class Window(C.Structure):
    _fields_ = [("k", _p), ("dim", C.c_int32), ("rope_dims", C.c_int32), ("rope_theta", C.c_float),
                ("format", C.c_int32), ("ring", _p), ("ring_scale", _p), ("ring_cap", C.c_int32),
                ("window_len", C.c_int32), ("ring_pages", C.POINTER(RingPages))]


class Query(C.Structure):
    _fields_ = [("q_in", _p), ("q_out", _p), ("gamma", _p), ("eps", C.c_float), ("num_heads", C.c_int32),
                ("dim", C.c_int32), ("rope_dims", C.c_int32), ("rope_theta", C.c_float)]


class IndexQuery(C.Structure):
    _fields_ = [("q_in", _p), ("q_out", _p), ("q_scale", _p), ("w_in", _p), ("w_out", _p), ("w_mult", C.c_float),
                ("num_heads", C.c_int32), ("dim", C.c_int32), ("rope_dims", C.c_int32), ("rope_theta", C.c_float)]


class CompressArgs(C.Structure):
    _fields_ = [("batch", Batch), ("main", C.POINTER(Compressor)), ("indexer", C.POINTER(Compressor)),
                ("window", C.POINTER(Window)), ("status", _p), ("query", C.POINTER(Query)),
                ("index_query", C.POINTER(IndexQuery))]


class IndexArgs(C.Structure):
    _fields_ = [("batch", Batch), ("keys", Cache), ("num_heads", C.c_int32), ("q_format", C.c_int32),
                ("q", _p), ("q_scale", _p), ("weights", _p), ("k", C.c_int32), ("out_idx", _p),
                ("status", _p)]


class AttnArgs(C.Structure):
    _fields_ = [("batch", Batch), ("kv", Cache), ("idx", _p), ("k", C.c_int32), ("window", _p),
                ("window_scale", _p), ("window_cap", C.c_int32), ("window_format", C.c_int32),
                ("window_len", C.c_int32), ("num_heads", C.c_int32), ("q", _p),
                ("softmax_scale", C.c_float), ("out", _p), ("lse", _p), ("status", _p),
                ("window_pages", C.POINTER(RingPages))]


class OutputArgs(C.Structure):
    _fields_ = [("num_tokens", C.c_int32), ("positions", _p), ("num_heads", C.c_int32),
                ("dim", C.c_int32), ("rope_dims", C.c_int32), ("rope_theta", C.c_float),
                ("in_", _p), ("out_format", C.c_int32), ("out", _p), ("out_scale", _p)]


_lib = None


def lib() -> C.CDLL:
    """The loaded libv4a; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libv4a.so not found at {LIB_PATH}: run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        L.v4a_compress_insert.argtypes = [C.POINTER(CompressArgs), _p]
        L.v4a_index_workspace_size.argtypes = [C.POINTER(IndexArgs)]
        L.v4a_index_workspace_size.restype = C.c_size_t
        L.v4a_index_topk.argtypes = [C.POINTER(IndexArgs), _p, C.c_size_t, _p]
        L.v4a_index_scores.argtypes = [C.POINTER(IndexArgs), _p, C.c_size_t, _p]
        L.v4a_index_select.argtypes = [C.POINTER(IndexArgs), _p, C.c_size_t, _p]
        L.v4a_index_topk_static.argtypes = [C.POINTER(IndexArgs), _p]
        L.v4a_index_scores_layout.argtypes = [C.POINTER(IndexArgs), C.POINTER(C.c_size_t),
                                              C.POINTER(C.c_int64)]
        L.v4a_attn_workspace_size.argtypes = [C.POINTER(AttnArgs)]
        L.v4a_attn_workspace_size.restype = C.c_size_t
        L.v4a_sparse_attn.argtypes = [C.POINTER(AttnArgs), _p, C.c_size_t, _p]
        L.v4a_inv_rope_quant.argtypes = [C.POINTER(OutputArgs), _p]
        L.v4a_sparse_attn_out.argtypes = [C.POINTER(AttnArgs), C.POINTER(OutputArgs), _p, C.c_size_t, _p]
        L.v4a_status_string.restype = C.c_char_p
        L.v4a_status_string.argtypes = [C.c_int]
        _lib = L
    return _lib


class V4AError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {lib().v4a_status_string(code).decode()} (code {code})")
        self.code = code


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(where: str, rc: int):
    if rc != V4A_OK:
        raise V4AError(where, rc)

# --------------------------------------------------------------------------
# Device-resident layer state
# --------------------------------------------------------------------------


@dataclass
class PagedViews:
    """Where a layer's caches and rings live when they are pages of shared
    bucket pools (pages.py): per cache (pool, pages in it, device table,
    table columns); per ring its v4a_ring_pages struct and capacity."""
    kv: tuple
    ix: tuple | None
    ring_main: RingPages | None
    main_cap: int
    ring_ix: RingPages | None
    ix_cap: int
    ring_swa: RingPages
    swa_cap: int


@dataclass
class DeviceLayer:
    """One layer's caches, rings, block table and the step inputs on the GPU
    (caches and rings in the layer's own tensors, or in shared page pools
    when `paged` is set)."""
    spec: object
    t: dict            # name -> CUDA tensor
    status: torch.Tensor
    paged: PagedViews | None = None

    @classmethod
    def from_case(cls, case, device="cuda") -> "DeviceLayer":
        t = {}
        for f in ("seq_ids", "positions", "block_table", "kv_pool", "x", "gate", "bias", "gamma",
                  "ring_x", "ring_gate", "k_swa", "swa_ring", "swa_scale", "q", "ix_pool", "x_i",
                  "gate_i", "bias_i", "gamma_i", "ring_x_i", "ring_gate_i", "q_i", "q_i_scale",
                  "w_i", "o_in", "q_raw", "gamma_q", "q_i_raw", "w_i_raw"):
            v = getattr(case, f)
            if v is not None and v.numel() > 0:
                t[f] = v.to(device).contiguous()
        if case.spec.window_only:
            # any non-NULL idx with k = 0 selects the window alone (never read)
            t["window_only_idx"] = torch.zeros(1, dtype=torch.int32, device=device)
        return cls(spec=case.spec, t=t, status=torch.zeros(1, dtype=torch.int32, device=device))

    # ---- argument structs -------------------------------------------------
    def batch(self) -> Batch:
        s = self.spec
        return Batch(s.tokens, _ptr(self.t["seq_ids"]), _ptr(self.t["positions"]), s.batch, s.new)

    def kv_cache(self) -> Cache:
        s = self.spec
        if self.paged:
            pool, n, table, cols = self.paged.kv
            return Cache(s.ratio, s.dim, s.rope_dims, s.theta, s.kv_fmt, _ptr(pool), n, _ptr(table), cols)
        return Cache(s.ratio, s.dim, s.rope_dims, s.theta, s.kv_fmt, _ptr(self.t["kv_pool"]),
                     s.num_blocks, _ptr(self.t["block_table"]), s.max_blocks)

    def ix_cache(self) -> Cache:
        s = self.spec
        if self.paged:
            pool, n, table, cols = self.paged.ix
            return Cache(4, s.ix_dim, s.ix_rope_dims, s.theta, s.ix_fmt, _ptr(pool), n, _ptr(table), cols)
        return Cache(4, s.ix_dim, s.ix_rope_dims, s.theta, s.ix_fmt, _ptr(self.t["ix_pool"]),
                     s.num_blocks, _ptr(self.t["block_table"]), s.max_blocks)

    def compress_args(self, parts=("main", "indexer", "window", "query", "index_query")):
        """Arguments of v4a_compress_insert for the named parts (the others
        NULL: the call skips them).  "query" (layers with q_prep) normalises
        and rotates q_raw into q, the attention's query; "index_query"
        (layers with ix_q_prep) rotates and encodes q_i_raw into q_i and
        q_i_scale and scales w_i_raw into w_i, the indexer's inputs."""
        s, t, pg = self.spec, self.t, self.paged
        keep = []
        main = ix = win = qry = ixq = None
        if "main" in parts:
            if pg:
                main = Compressor(self.kv_cache(), _ptr(t["x"]), _ptr(t["gate"]), _ptr(t["bias"]),
                                  _ptr(t["gamma"]), 1e-6, None, None, pg.main_cap, C.pointer(pg.ring_main))
            else:
                main = Compressor(self.kv_cache(), _ptr(t["x"]), _ptr(t["gate"]), _ptr(t["bias"]),
                                  _ptr(t["gamma"]), 1e-6, _ptr(t["ring_x"]), _ptr(t["ring_gate"]), s.ring_cap)
            keep.append(main)
        if s.ix_heads and "indexer" in parts:
            if pg:
                ix = Compressor(self.ix_cache(), _ptr(t["x_i"]), _ptr(t["gate_i"]), _ptr(t["bias_i"]),
                                _ptr(t["gamma_i"]), 1e-6, None, None, pg.ix_cap, C.pointer(pg.ring_ix))
            else:
                ix = Compressor(self.ix_cache(), _ptr(t["x_i"]), _ptr(t["gate_i"]), _ptr(t["bias_i"]),
                                _ptr(t["gamma_i"]), 1e-6, _ptr(t["ring_x_i"]), _ptr(t["ring_gate_i"]),
                                s.ix_ring_cap)
            keep.append(ix)
        if "window" in parts:
            if pg:
                win = Window(_ptr(t["k_swa"]), s.dim, s.rope_dims, s.theta, s.swa_fmt, None, None, pg.swa_cap,
                             s.swa, C.pointer(pg.ring_swa))
            else:
                win = Window(_ptr(t["k_swa"]), s.dim, s.rope_dims, s.theta, s.swa_fmt, _ptr(t["swa_ring"]),
                             _ptr(t.get("swa_scale")), s.swa_cap, s.swa)
            keep.append(win)
        if s.q_prep and "query" in parts:
            qry = Query(_ptr(t["q_raw"]), _ptr(t["q"]), _ptr(t["gamma_q"]), 1e-6, s.heads, s.dim, s.rope_dims,
                        s.theta)
            keep.append(qry)
        if s.ix_q_prep and "index_query" in parts:
            ixq = IndexQuery(_ptr(t["q_i_raw"]), _ptr(t["q_i"]), _ptr(t["q_i_scale"]), _ptr(t["w_i_raw"]),
                             _ptr(t["w_i"]), s.ix_w_mult, s.ix_heads, s.ix_dim, s.ix_rope_dims, s.theta)
            keep.append(ixq)
        a = CompressArgs(self.batch(), C.pointer(main) if main else None, C.pointer(ix) if ix else None,
                         C.pointer(win) if win else None, _ptr(self.status), C.pointer(qry) if qry else None,
                         C.pointer(ixq) if ixq else None)
        return a, keep

    def index_args(self, out_idx: torch.Tensor) -> IndexArgs:
        s, t = self.spec, self.t
        return IndexArgs(self.batch(), self.ix_cache(), s.ix_heads, s.ix_q_fmt, _ptr(t["q_i"]),
                         _ptr(t["q_i_scale"]), _ptr(t["w_i"]), s.topk, _ptr(out_idx),
                         _ptr(self.status))

    def attn_args(self, idx: torch.Tensor | None, out: torch.Tensor, lse: torch.Tensor | None) -> AttnArgs:
        s, t = self.spec, self.t
        if s.window_only:
            idx, k = t["window_only_idx"], 0
        else:
            k = s.topk if idx is not None else 0
        if self.paged:
            pg = self.paged
            return AttnArgs(self.batch(), self.kv_cache(), _ptr(idx), k, None, None, pg.swa_cap, s.swa_fmt,
                            s.swa, s.heads, _ptr(t["q"]), 1.0 / math.sqrt(s.dim), _ptr(out), _ptr(lse),
                            _ptr(self.status), C.pointer(pg.ring_swa))
        return AttnArgs(self.batch(), self.kv_cache(), _ptr(idx), k,
                        _ptr(t["swa_ring"]), _ptr(t.get("swa_scale")), s.swa_cap, s.swa_fmt, s.swa,
                        s.heads, _ptr(t["q"]), 1.0 / math.sqrt(s.dim), _ptr(out), _ptr(lse),
                        _ptr(self.status))

    def output_args(self, o: torch.Tensor, out: torch.Tensor, out_scale: torch.Tensor | None) -> OutputArgs:
        s = self.spec
        return OutputArgs(s.tokens, _ptr(self.t["positions"]), s.heads, s.dim, s.rope_dims, s.theta,
                          _ptr(o), s.out_fmt, _ptr(out), _ptr(out_scale))

# --------------------------------------------------------------------------
# Calls
# --------------------------------------------------------------------------


def compress_insert(layer: DeviceLayer, stream=None, parts=("main", "indexer", "window", "query", "index_query")):
    a, keep = layer.compress_args(parts)
    _check("v4a_compress_insert", lib().v4a_compress_insert(C.byref(a), _stream(stream)))


def index_workspace_bytes(layer: DeviceLayer) -> int:
    out = torch.empty(0, dtype=torch.int32)
    a = layer.index_args(out)
    return int(lib().v4a_index_workspace_size(C.byref(a)))


def index_topk(layer: DeviceLayer, out_idx: torch.Tensor, workspace: torch.Tensor, stream=None):
    a = layer.index_args(out_idx)
    _check("v4a_index_topk", lib().v4a_index_topk(C.byref(a), _ptr(workspace), workspace.numel(),
                                                  _stream(stream)))


# Scratch limit of v4a_index_topk_static (V4A_INDEX_STATIC_SCRATCH_BYTES in v4a.h).
INDEX_STATIC_SCRATCH_BYTES = 16 << 20


def index_topk_static(layer: DeviceLayer, out_idx: torch.Tensor, stream=None):
    """v4a_index_topk with the library's fixed device scratch: no workspace is
    passed, nothing is allocated (for callers that may not allocate)."""
    a = layer.index_args(out_idx)
    _check("v4a_index_topk_static", lib().v4a_index_topk_static(C.byref(a), _stream(stream)))


def index_scores(layer: DeviceLayer, out_idx: torch.Tensor, workspace: torch.Tensor, stream=None):
    a = layer.index_args(out_idx)
    _check("v4a_index_scores", lib().v4a_index_scores(C.byref(a), _ptr(workspace), workspace.numel(),
                                                      _stream(stream)))


def index_select(layer: DeviceLayer, out_idx: torch.Tensor, workspace: torch.Tensor, stream=None):
    a = layer.index_args(out_idx)
    _check("v4a_index_select", lib().v4a_index_select(C.byref(a), _ptr(workspace), workspace.numel(),
                                                      _stream(stream)))


def index_scores_view(layer: DeviceLayer, workspace: torch.Tensor) -> torch.Tensor:
    """The [T][row] fp32 score matrix that v4a_index_scores left in `workspace`."""
    a = layer.index_args(torch.empty(0, dtype=torch.int32))
    off, row = C.c_size_t(), C.c_int64()
    _check("v4a_index_scores_layout", lib().v4a_index_scores_layout(C.byref(a), C.byref(off), C.byref(row)))
    T = layer.spec.tokens
    return workspace[off.value: off.value + 4 * T * row.value].view(torch.float32).view(T, row.value)


def attn_workspace_bytes(layer: DeviceLayer, with_idx: bool) -> int:
    dummy = torch.empty(0, dtype=torch.int32)
    a = layer.attn_args(dummy if with_idx else None, dummy, None)
    if with_idx:
        a.idx = 1   # any non-null value: only the presence matters for sizing
    return int(lib().v4a_attn_workspace_size(C.byref(a)))


def sparse_attn(layer: DeviceLayer, idx: torch.Tensor | None, out: torch.Tensor,
                lse: torch.Tensor | None, workspace: torch.Tensor, stream=None):
    a = layer.attn_args(idx, out, lse)
    _check("v4a_sparse_attn", lib().v4a_sparse_attn(C.byref(a), _ptr(workspace), workspace.numel(),
                                                    _stream(stream)))


def inv_rope_quant(layer: DeviceLayer, o: torch.Tensor, out: torch.Tensor,
                   out_scale: torch.Tensor | None, stream=None):
    a = layer.output_args(o, out, out_scale)
    _check("v4a_inv_rope_quant", lib().v4a_inv_rope_quant(C.byref(a), _stream(stream)))


V4A_ERR_UNSUPPORTED = 2


def sparse_attn_out(layer: DeviceLayer, idx: torch.Tensor | None, out: torch.Tensor,
                    out_scale: torch.Tensor | None, workspace: torch.Tensor, stream=None) -> bool:
    """Attention + inverse RoPE + output encode in one call (the bf16 attention
    output is not stored).  False, with nothing launched, when the shapes are
    outside the fused path; any other failure raises."""
    a = layer.attn_args(idx, None, None)
    o = layer.output_args(None, out, out_scale)
    rc = lib().v4a_sparse_attn_out(C.byref(a), C.byref(o), _ptr(workspace), workspace.numel(), _stream(stream))
    if rc == V4A_ERR_UNSUPPORTED:
        return False
    _check("v4a_sparse_attn_out", rc)
    return True


class Step:
    """Output buffers + workspaces for running whole layer steps on a DeviceLayer.

    fused_out: attention and output stage as one call (v4a_sparse_attn_out)
    where the library takes the shapes; self.o is then not written.

    overlap: how the compressor calls are placed (layers with an indexer):
      "serial"  one compress call (all parts), then the indexer, attention;
      "start"   the indexer pipeline (indexer compressor -> scan -> top-k) on
                the calling stream and the main compressor + window insert on
                a side stream from the start of the step, joined before the
                attention (the pages' separate indexer stream);
      "select"  as "start", with the side-stream call placed after the scan,
                where it runs beside the top-k (which leaves most SMs idle)
                instead of beside the scan (which holds every SM)."""

    def __init__(self, layer: DeviceLayer, fused_out: bool = True, overlap: str = "serial"):
        s = layer.spec
        dev = layer.status.device
        self.layer = layer
        self.fused_out = fused_out
        assert overlap in ("serial", "start", "select")
        self.overlap = overlap if s.ix_heads else "serial"
        self.side = torch.cuda.Stream(device=dev) if self.overlap != "serial" else None
        T = s.tokens
        self.idx = torch.full((T, s.topk), -1, dtype=torch.int32, device=dev) if s.ix_heads else None
        self.o = torch.empty((T, s.heads, s.dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, s.heads), dtype=torch.float32, device=dev)
        if s.out_fmt == OUT_BF16:
            self.out = torch.empty((T, s.heads, s.dim), dtype=torch.bfloat16, device=dev)
            self.out_scale = None
        else:
            self.out = torch.empty((T, s.heads, s.dim), dtype=torch.uint8, device=dev)
            self.out_scale = torch.empty((T,), dtype=torch.float32, device=dev)
        self.ws_index = torch.empty(max(index_workspace_bytes(layer) if s.ix_heads else 0, 256),
                                    dtype=torch.uint8, device=dev)
        self.ws_attn = torch.empty(max(attn_workspace_bytes(layer, s.ix_heads > 0), 256),
                                   dtype=torch.uint8, device=dev)

    def launches_per_step(self) -> int:
        """libv4a kernels one run() launches: compress (1, 2 when split over
        two streams); indexer workspace clear (1) + scan (1) + top-k (1, plus
        the histogram kernel for long rows scored on the CUDA cores); then per
        batch of queries either attention + merge + encode (fused output) or
        attention (+ combine when the key list is split) and the output stage."""
        s = self.layer.spec
        n = 1 if self.overlap == "serial" else 2   # compress (split in two with overlap)
        if s.ix_heads:
            tc_scan = s.ix_fmt in (IX_FP8_B128, IX_FP4_B32, IX_FP4_MX32) and s.ix_heads == 64 and s.ix_dim == 128
            # clear + scan, then the top-k: one kernel (plus the histogram
            # kernel for long rows scored on the CUDA cores)
            n += 2 + (1 if s.max_blocks * 64 <= 32768 or tc_scan else 2)
        # the tensor-core attention runs long batches (chunked prefill) as
        # several launches of at most 64 waves of 152 CTAs, one CTA per
        # 64-key chunk of a query's list
        nsel = 0 if s.window_only else (s.topk if s.ix_heads else s.max_blocks * (256 // s.ratio))
        chunks = -(-(nsel + s.swa) // 64)
        per = max(1, min(s.tokens, (64 * 152) // chunks))
        batches = -(-s.tokens // per)
        if self.fused_out:
            return n + 3 * batches            # attention, merge and encode kernels per batch
        n += batches * (1 + (1 if chunks > 1 else 0))
        return n + 1

    def run(self, stream=None):
        """compress_insert -> index_topk -> sparse_attn -> inv_rope_quant
        (with `overlap`, the compressor's parts split over two streams)."""
        L = self.layer
        if L.spec.window_only:
            compress_insert(L, stream, parts=("window", "query"))   # a pure sliding-window layer has no compressor
        elif self.overlap == "serial":
            compress_insert(L, stream)
            if L.spec.ix_heads:
                index_topk(L, self.idx, self.ws_index, stream)
        else:
            cur = stream if stream is not None else torch.cuda.current_stream()
            fork = torch.cuda.Event()
            joined = torch.cuda.Event()
            fork.record(cur)
            compress_insert(L, cur, parts=("indexer", "index_query"))
            if self.overlap == "select":
                index_scores(L, self.idx, self.ws_index, cur)
                fork.record(cur)
            self.side.wait_event(fork)
            compress_insert(L, self.side, parts=("main", "window", "query"))
            joined.record(self.side)
            if self.overlap == "select":
                index_select(L, self.idx, self.ws_index, cur)
            else:
                index_topk(L, self.idx, self.ws_index, cur)
            cur.wait_event(joined)
        if self.fused_out:
            if sparse_attn_out(L, self.idx, self.out, self.out_scale, self.ws_attn, stream):
                return
            self.fused_out = False            # shapes outside the fused path: the two calls
        sparse_attn(L, self.idx, self.o, self.lse, self.ws_attn, stream)
        inv_rope_quant(L, self.o, self.out, self.out_scale, stream)
