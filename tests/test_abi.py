"""The C-ABI library loads on a machine without a GPU, exports every entry
point the header declares, and rejects bad arguments on the host (no GPU
call is made on these paths)."""
import ctypes as C
import os
import re

import pytest

from compressed_sparse_long_c4a_gb300 import inputs as I
from compressed_sparse_long_c4a_gb300 import v4a

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(v4a.LIB_PATH):
        from compressed_sparse_long_c4a_gb300 import build
        build.build()
    return v4a.lib()


def test_exports_every_declared_symbol(lib):
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            hdr = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"V4A_API\s+[\w\s\*]+?\b(v4a_\w+)\s*\(", hdr)
    assert len(names) >= 18 and "v4a_pages_create" in names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.v4a_abi_version() == 5
    for code in range(7):
        assert lib.v4a_status_string(code).decode() != "unknown status"


class _FakeLayer(v4a.DeviceLayer):
    """Argument structs with fake (never dereferenced) device pointers."""

    def __init__(self, spec):
        self.spec = spec
        self.t = {}
        self.status = None

    def batch(self):
        s = self.spec
        return v4a.Batch(s.tokens, 0x1000, 0x2000, s.batch, s.new)

    def kv_cache(self):
        s = self.spec
        return v4a.Cache(s.ratio, s.dim, s.rope_dims, s.theta, s.kv_fmt, 0x3000, s.num_blocks, 0x4000,
                         s.max_blocks)

    def ix_cache(self):
        s = self.spec
        return v4a.Cache(4, s.ix_dim, s.ix_rope_dims, s.theta, s.ix_fmt, 0x5000, s.num_blocks, 0x4000,
                         s.max_blocks)


def _compressor(layer, cap):
    return v4a.Compressor(layer.kv_cache(), 0x10, 0x20, 0x30, 0x40, 1e-6, 0x50, 0x60, cap)


def test_host_validation_of_compress(lib):
    spec = I.c4a_prefill_4x4k()
    L = _FakeLayer(spec)
    assert lib.v4a_compress_insert(None, None) == 1
    comp = _compressor(L, spec.ring_cap - 1)           # one slot short: window - 2 + new
    a = v4a.CompressArgs(L.batch(), C.pointer(comp), None, None, None)
    assert lib.v4a_compress_insert(C.byref(a), None) == 3
    win = v4a.Window(0x70, spec.dim, 64, 1e4, 0, 0x80, None, 127 + spec.new - 1, 128)
    a = v4a.CompressArgs(L.batch(), None, None, C.pointer(win), None)
    assert lib.v4a_compress_insert(C.byref(a), None) == 3             # one slot short of window - 1 + new
    # the bound follows the window length: an empty batch validates and
    # launches nothing, so these calls reach no device
    b0 = L.batch()
    b0.num_tokens = 0
    a0 = v4a.CompressArgs(b0, None, None, C.pointer(win), None)
    win.ring_cap, win.window_len = 64 + spec.new - 1, 64
    assert lib.v4a_compress_insert(C.byref(a0), None) == 0
    win.ring_cap = 64 + spec.new - 2
    assert lib.v4a_compress_insert(C.byref(a0), None) == 3
    win.window_len = 0
    assert lib.v4a_compress_insert(C.byref(a0), None) == 1
    bad = _compressor(L, spec.ring_cap)
    bad.cache.ratio = 5
    a = v4a.CompressArgs(L.batch(), C.pointer(bad), None, None, None)
    assert lib.v4a_compress_insert(C.byref(a), None) == 1
    odd = _compressor(L, spec.ring_cap)
    odd.cache.dim = 96
    a = v4a.CompressArgs(L.batch(), C.pointer(odd), None, None, None)
    assert lib.v4a_compress_insert(C.byref(a), None) == 2


def test_host_validation_of_index_and_workspace_sizes(lib):
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    a = v4a.IndexArgs(L.batch(), L.ix_cache(), spec.ix_heads, spec.ix_q_fmt, 0x10, 0x20, 0x30, spec.topk,
                      0x40, None)
    need = lib.v4a_index_workspace_size(C.byref(a))
    # scores for every visible entry of every query at least
    assert need >= spec.tokens * spec.max_blocks * 64 * 4
    assert lib.v4a_index_topk(C.byref(a), None, 0, None) == 4           # no workspace
    assert lib.v4a_index_topk(C.byref(a), 0x1000, need - 1, None) == 4
    a.k = 0
    assert lib.v4a_index_topk(C.byref(a), 0x1000, need, None) == 2
    a.k = spec.topk
    a.q_format = v4a.Q_BF16                                              # fp4 keys need an fp8 query
    assert lib.v4a_index_topk(C.byref(a), 0x1000, need, None) == 2
    a.q_format = v4a.Q_FP8_HEAD
    a.keys.ratio = 128
    assert lib.v4a_index_topk(C.byref(a), 0x1000, need, None) == 2


def test_host_validation_of_attention_and_output(lib):
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    a = v4a.AttnArgs(L.batch(), L.kv_cache(), 0x10, spec.topk, 0x20, 0x30, spec.swa_cap, spec.swa_fmt,
                     spec.swa, spec.heads, 0x40, 0.04, 0x50, None, None)
    need = lib.v4a_attn_workspace_size(C.byref(a))
    assert need > 0
    assert lib.v4a_sparse_attn(C.byref(a), None, 0, None) == 4
    a.window_scale = None                                                # fp8 window needs scales
    assert lib.v4a_sparse_attn(C.byref(a), 0x1000, need, None) == 1
    a.window_scale = 0x30
    a.window_cap = spec.swa - 2 + spec.new                               # one slot short of window - 1 + new
    assert lib.v4a_sparse_attn(C.byref(a), 0x1000, need, None) == 3
    a.window_cap = spec.swa_cap
    a.kv.dim = 96
    assert lib.v4a_sparse_attn(C.byref(a), 0x1000, need, None) == 2
    o = v4a.OutputArgs(4, 0x10, 128, 512, 64, 1e4, 0x20, 1, 0x30, None)  # fp8 output needs scales
    assert lib.v4a_inv_rope_quant(C.byref(o), None) == 1
    o = v4a.OutputArgs(0, None, 128, 512, 64, 1e4, None, 0, None, None)  # empty batch: no work
    assert lib.v4a_inv_rope_quant(C.byref(o), None) == 0


def test_host_validation_of_fused_attention_output(lib):
    """v4a_sparse_attn_out rejects bad or mismatched arguments before any
    device call (the checks come before the cluster-size query)."""
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    a = v4a.AttnArgs(L.batch(), L.kv_cache(), 0x10, spec.topk, 0x20, 0x30, spec.swa_cap, spec.swa_fmt,
                     spec.swa, spec.heads, 0x40, 0.04, None, None, None)
    o = v4a.OutputArgs(spec.tokens, 0x2000, spec.heads, spec.dim, spec.rope_dims, spec.theta, None,
                       spec.out_fmt, 0x60, 0x70)
    assert lib.v4a_sparse_attn_out(None, C.byref(o), 0x1000, 1 << 30, None) == 1
    assert lib.v4a_sparse_attn_out(C.byref(a), None, 0x1000, 1 << 30, None) == 1
    o.num_tokens = spec.tokens + 1                                        # not the attention's tokens
    assert lib.v4a_sparse_attn_out(C.byref(a), C.byref(o), 0x1000, 1 << 30, None) == 1
    o.num_tokens = spec.tokens
    o.num_heads = spec.heads // 2                                         # not the attention's heads
    assert lib.v4a_sparse_attn_out(C.byref(a), C.byref(o), 0x1000, 1 << 30, None) == 1
    o.num_heads = spec.heads
    o.out_format = 7
    assert lib.v4a_sparse_attn_out(C.byref(a), C.byref(o), 0x1000, 1 << 30, None) == 1
    o.out_format = spec.out_fmt
    o.out_scale = None                                                    # fp8 output needs its scales
    assert lib.v4a_sparse_attn_out(C.byref(a), C.byref(o), 0x1000, 1 << 30, None) == 1


def test_attention_workspace_covers_one_launch_of_a_long_batch(lib):
    """Chunked prefill (16,384 queries, 10 key chunks each) runs as several
    launches that reuse one launch's worth of chunk results: the workspace is
    sized for at most 64 waves of 152 CTAs, not for the whole batch."""
    spec = I.c4a_prefill_4x4k()
    L = _FakeLayer(spec)
    a = v4a.AttnArgs(L.batch(), L.kv_cache(), 0x10, spec.topk, 0x20, 0x30, spec.swa_cap, spec.swa_fmt,
                     spec.swa, spec.heads, 0x40, 0.04, 0x50, None, None)
    need = lib.v4a_attn_workspace_size(C.byref(a))
    chunks = -(-(spec.topk + spec.swa) // 64)
    per_launch = (64 * 152) // chunks
    row = chunks * spec.heads * (spec.dim * 2 + 8)          # bf16 row + (max, sum) per chunk and head
    assert spec.tokens > per_launch                          # the batch needs several launches
    assert per_launch * row <= need < 2 * per_launch * row
    # a decode batch fits one launch: its workspace covers every query
    d = I.c4a_decode_1m()
    Ld = _FakeLayer(d)
    ad = v4a.AttnArgs(Ld.batch(), Ld.kv_cache(), 0x10, d.topk, 0x20, 0x30, d.swa_cap, d.swa_fmt,
                      d.swa, d.heads, 0x40, 0.04, 0x50, None, None)
    dchunks = -(-(d.topk + d.swa) // 64)
    assert lib.v4a_attn_workspace_size(C.byref(ad)) >= d.tokens * dchunks * d.heads * (d.dim * 2 + 8)


def test_host_validation_of_paged_rings(lib):
    """A ring kept in pages must name a 16-byte aligned pool and page stride,
    a capacity that is a whole number of pages and pages large enough for
    their slots (row + fp32); an empty batch checks them without launching."""
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    b0 = L.batch()
    b0.num_tokens = 0
    cap = 32 * 4                                   # >= window - 1 + new for the c4a compressor
    row = 2 * spec.dim + 4

    def run(pool=0x10000, page_bytes=32 * row, slots=32, cap=cap, table=0x9000):
        rp = v4a.RingPages(pool, 1000, page_bytes, table, slots)
        comp = v4a.Compressor(L.kv_cache(), 0x10, 0x20, 0x30, 0x40, 1e-6, None, None, cap, C.pointer(rp))
        a = v4a.CompressArgs(b0, C.pointer(comp), None, None, None)
        return lib.v4a_compress_insert(C.byref(a), None)

    assert 32 * row % 16 == 0
    assert run() == 0
    assert run(page_bytes=32 * row - 16) == 1      # too small for 32 slots
    assert run(page_bytes=32 * row + 8) == 1       # stride not a multiple of 16
    assert run(pool=0x10008) == 1                  # pool not 16-byte aligned
    assert run(cap=cap + 1) == 1                   # capacity not a whole number of pages
    assert run(table=None) == 1
    # the window ring: fp8 rows carry an fp32 scale, bf16 rows none
    for fmt, rb in ((I.KV_FP8_TOKEN, spec.dim + 4), (I.KV_BF16, 2 * spec.dim)):
        for pb, want in ((64 * rb + (-64 * rb) % 16, 0), (64 * rb - 16, 1)):
            rp = v4a.RingPages(0x10000, 100, pb, 0x9000, 64)
            win = v4a.Window(0x70, spec.dim, 64, 1e4, fmt, None, None, 128 * 2, 128, C.pointer(rp))
            a = v4a.CompressArgs(b0, None, None, C.pointer(win), None)
            assert lib.v4a_compress_insert(C.byref(a), None) == want, (fmt, pb)


def test_host_validation_of_query_part(lib):
    """The queries' norm + RoPE part: pointers, a dim that is a multiple of 64
    up to 1024, even rope dims up to 128; checked with an empty batch."""
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    b0 = L.batch()
    b0.num_tokens = 0

    def run(q_in=0x100, q_out=0x200, gamma=0x300, heads=128, dim=512, rope=64, eps=1e-6):
        q = v4a.Query(q_in, q_out, gamma, eps, heads, dim, rope, 1e4)
        a = v4a.CompressArgs(b0, None, None, None, None, C.pointer(q))
        return lib.v4a_compress_insert(C.byref(a), None)

    assert run() == 0
    assert run(q_out=0x100) == 0            # in place
    assert run(q_in=None) == 1 and run(q_out=None) == 1 and run(gamma=None) == 1
    assert run(heads=0) == 1
    assert run(dim=96) == 2 and run(dim=2048) == 2
    assert run(rope=63) == 1 and run(rope=600) == 1 and run(rope=256) == 2
    assert run(eps=-1.0) == 1


def test_host_validation_of_index_query_part(lib):
    """The indexer query's RoPE + fp8 + weights part: every pointer, a dim
    that is a multiple of 64 up to 1024, even rope dims up to 128."""
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    b0 = L.batch()
    b0.num_tokens = 0

    def run(q_in=0x100, q_out=0x200, q_scale=0x300, w_in=0x400, w_out=0x500, heads=64, dim=128, rope=64):
        q = v4a.IndexQuery(q_in, q_out, q_scale, w_in, w_out, 0.5, heads, dim, rope, 1e4)
        a = v4a.CompressArgs(b0, None, None, None, None, None, C.pointer(q))
        return lib.v4a_compress_insert(C.byref(a), None)

    assert run() == 0 and run(w_out=0x400) == 0        # weights in place
    for k in ("q_in", "q_out", "q_scale", "w_in", "w_out"):
        assert run(**{k: None}) == 1, k
    assert run(heads=0) == 1
    assert run(dim=96) == 2 and run(dim=2048) == 2
    assert run(rope=63) == 1 and run(rope=256) == 1 and run(dim=512, rope=256) == 2


def test_misaligned_rows_are_refused_before_launch(lib):
    """Row pointers the compressor launch reads or writes in pairs must be
    aligned to the pair's width; a misaligned one is an invalid argument
    (checked on the host with an empty batch, so nothing launches)."""
    spec = I.c4a_decode_1m()
    L = _FakeLayer(spec)
    b0 = L.batch()
    b0.num_tokens = 0
    comp = v4a.Compressor(L.kv_cache(), 0x12, 0x20, 0x30, 0x40, 1e-6, 0x50, 0x60, 32)   # x on 2 bytes
    assert lib.v4a_compress_insert(C.byref(v4a.CompressArgs(b0, C.pointer(comp), None, None, None)), None) == 1
    comp.x = 0x10
    assert lib.v4a_compress_insert(C.byref(v4a.CompressArgs(b0, C.pointer(comp), None, None, None)), None) == 0
    win = v4a.Window(0x72, spec.dim, 64, 1e4, 0, 0x80, None, 128, 128)                  # k on 2 bytes
    assert lib.v4a_compress_insert(C.byref(v4a.CompressArgs(b0, None, None, C.pointer(win), None)), None) == 1
    q = v4a.Query(0x100, 0x200, 0x304, 1e-6, 128, 512, 64, 1e4)                         # gamma on 4 bytes
    assert lib.v4a_compress_insert(C.byref(v4a.CompressArgs(b0, None, None, None, None, C.pointer(q))), None) == 1
    q.gamma = 0x308
    assert lib.v4a_compress_insert(C.byref(v4a.CompressArgs(b0, None, None, None, None, C.pointer(q))), None) == 0
    iq = v4a.IndexQuery(0x100, 0x201, 0x300, 0x400, 0x500, 0.5, 64, 128, 64, 1e4)        # codes on 1 byte
    a = v4a.CompressArgs(b0, None, None, None, None, None, C.pointer(iq))
    assert lib.v4a_compress_insert(C.byref(a), None) == 1
    iq.q_out = 0x202
    assert lib.v4a_compress_insert(C.byref(a), None) == 0


def test_attention_refuses_misaligned_key_rows(lib):
    """Cache and window rows are read as 4-byte words: a pool or window that
    does not start on 4 bytes is an invalid argument, refused before any
    launch."""
    spec = I.c4a_decode_1k()
    L = _FakeLayer(spec)
    kv = L.kv_cache()
    kv.pool = 0x3002
    a = v4a.AttnArgs(L.batch(), kv, 0x9000, spec.topk, 0x7000, None, spec.swa_cap, spec.swa_fmt, spec.swa,
                     spec.heads, 0xA000, 0.1, 0xB000, None, None)
    assert lib.v4a_sparse_attn(C.byref(a), 0xC000, 1 << 30, None) == 1
    a.kv.pool, a.window = 0x3000, 0x7002
    assert lib.v4a_sparse_attn(C.byref(a), 0xC000, 1 << 30, None) == 1
