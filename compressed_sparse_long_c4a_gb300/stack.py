"""A model's attention layers as one step: every layer's compress -> indexer
-> attention -> output path, in layer order, replayed from one CUDA graph.

Source: "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
(the layer mix: c4a layers with the indexer, c128a layers that attend to
every compressed entry, and layers that use the sliding window alone) and
Appendix "the arithmetic behind 8.7x" (61 attention layers: 30 c4a and 31
c128a); CUDA Graphs in "keeping the GPU busy".

Readings: the pages give the counts of c4a and c128a layers but neither
their order nor the number of pure sliding-window layers.  `deepseek_v4_mix`
alternates them starting with c128a (31 + 30 = 61) and takes the number of
window-only layers as a parameter (0 in the 61-layer count).

Each layer has its own caches, rings and workspaces (built from one synthetic
case per layer kind and copied per layer), so a replay of the graph is one
decode step of the whole attention stack: every layer inserts its new
entries and attends over its own caches.  With paged=True the caches and
rings of all layers are pages of one device pool per page-size bucket, handed
out by the library's page allocator ("keeping the KV cache memory packed" on
the same page: c4a KV, SWA KV and both compressor states in the largest
bucket, the indexer KV and the indexer's state in the middle one, c128a KV in
the smallest).
"""
from __future__ import annotations

import collections
import dataclasses

import numpy as np
import torch

from . import inputs as I
from . import pages as P
from . import v4a

# step inputs a layer keeps in its own tensors when its caches and rings are paged
_STEP_INPUTS = ("seq_ids", "positions", "x", "gate", "bias", "gamma", "k_swa", "q", "x_i", "gate_i",
                "bias_i", "gamma_i", "q_i", "q_i_scale", "w_i", "o_in", "window_only_idx", "q_raw", "gamma_q", "q_i_raw", "w_i_raw")


def deepseek_v4_mix(n_c4a: int = 30, n_c128a: int = 31, n_swa: int = 0) -> list:
    """Layer kinds in order: c128a and c4a alternating (c128a first) while
    both last, then the remainder, then the window-only layers."""
    kinds = []
    a, b = n_c128a, n_c4a
    while a or b:
        if a:
            kinds.append("c128a")
            a -= 1
        if b:
            kinds.append("c4a")
            b -= 1
    return kinds + ["swa"] * n_swa


class AttentionStack:
    """Layers of the given kinds ("c4a", "c128a", "swa") built from one case
    per kind (`cases`, keyed by kind), each layer with its own device copies."""

    def __init__(self, kinds: list, cases: dict, device="cuda", overlap: str = "serial", paged: bool = False):
        self.kinds = list(kinds)
        self.layers = []
        self.steps = []
        self.alloc = None
        self.pools = []
        proto = {}
        for k in set(self.kinds):
            proto[k] = v4a.DeviceLayer.from_case(cases[k], device)
        if paged:
            self._build_paged(cases, proto, device)
        else:
            for k in self.kinds:
                p = proto[k]
                self.layers.append(v4a.DeviceLayer(spec=p.spec, t={n: x.clone() for n, x in p.t.items()},
                                                   status=torch.zeros(1, dtype=torch.int32, device=device)))
        for k, L in zip(self.kinds, self.layers):
            self.steps.append(v4a.Step(L, overlap=overlap if k == "c4a" else "serial"))
        del proto

    # ---- caches and rings in page-size buckets ----------------------------------
    def _build_paged(self, cases: dict, proto: dict, device):
        specs = {k: cases[k].spec for k in set(self.kinds)}
        s0 = specs[self.kinds[0]]
        for s in specs.values():
            # one context per sequence in every layer
            if (s.batch, s.cached, s.new) != (s0.batch, s0.cached, s0.new):
                raise ValueError("paged stack: every layer kind needs the same batch, cached and new")
        count = collections.Counter(self.kinds)
        sizes = []
        if "c4a" in count:
            sizes += [specs["c4a"].kv_block_bytes, specs["c4a"].ix_block_bytes]
        if "c128a" in count:
            sizes.append(specs["c128a"].kv_block_bytes)
        if not sizes:
            raise ValueError("paged stack: no compressed cache to size the pages")
        ranks = sorted(set(sizes), reverse=True)
        # rings join the c4a KV bucket (the largest), the indexer's state the indexer KV bucket
        main_rank = ranks.index(specs["c4a"].kv_block_bytes) if "c4a" in count else 0
        kinds, slot = [], {}

        def add(name, k):
            slot[name] = len(kinds)
            kinds.append(k)

        def swa_slot(s):
            return 2 * s.dim if s.swa_fmt == I.KV_BF16 else s.dim + 4

        if "c4a" in count:
            s, n = specs["c4a"], count["c4a"]
            add("c4a.kv", P.block_kind(s.kv_block_bytes, n))
            add("c4a.ix", P.block_kind(s.ix_block_bytes, n))
            add("c4a.state", P.ring_kind(2 * s.dim + 4, s.ring_cap, main_rank, n))
            add("c4a.ix_state", P.ring_kind(2 * s.ix_dim + 4, s.ix_ring_cap, ranks.index(s.ix_block_bytes), n))
            add("c4a.swa", P.ring_kind(swa_slot(s), s.swa_cap, main_rank, n))
        if "c128a" in count:
            s, n = specs["c128a"], count["c128a"]
            add("c128a.kv", P.block_kind(s.kv_block_bytes, n))
            add("c128a.state", P.ring_kind(2 * s.dim + 4, s.ring_cap, main_rank, n))
            add("c128a.swa", P.ring_kind(swa_slot(s), s.swa_cap, main_rank, n))
        if "swa" in count:
            s, n = specs["swa"], count["swa"]
            add("swa.swa", P.ring_kind(swa_slot(s), s.swa_cap, main_rank, n))
        # the pools hold as many logical blocks as the tables address
        B = s0.batch
        alloc = P.PageAllocator(kinds, B, s0.max_blocks, budget_bytes=1 << 60)
        for b in range(B):
            alloc.open(b)
            alloc.reserve(b, s0.cached[b] + s0.new)
        buckets = alloc.buckets()
        self.alloc, self.slot = alloc, slot
        self.pools = [torch.zeros(bk.num_pages * bk.page_bytes, dtype=torch.uint8, device=device)
                      for bk in buckets]
        self.tables = torch.from_numpy(alloc.tables().copy()).to(device)
        self._dummy_table = torch.full((B, 1), -1, dtype=torch.int32, device=device)
        seen = collections.Counter()
        for k in self.kinds:
            li = seen[k]
            seen[k] += 1
            p = proto[k]
            case = cases[k]
            t = {n: p.t[n].clone() for n in _STEP_INPUTS if n in p.t}
            if k == "swa":
                kv = (self.pools[0], buckets[0].num_pages, self._dummy_table, 1)   # never read
            else:
                kv = self._paged_cache(f"{k}.kv", li, p.t["kv_pool"], case.block_table)
            ix = ring_main = ring_ix = None
            main_cap = ix_cap = 0
            if k == "c4a":
                ix = self._paged_cache("c4a.ix", li, p.t["ix_pool"], case.block_table)
                ring_ix, ix_cap = self._paged_ring("c4a.ix_state", li, p.t["ring_x_i"], p.t["ring_gate_i"],
                                                   case.spec)
            if k != "swa":
                ring_main, main_cap = self._paged_ring(f"{k}.state", li, p.t["ring_x"], p.t["ring_gate"],
                                                       case.spec)
            ring_swa, swa_cap = self._paged_ring(f"{k}.swa", li, p.t["swa_ring"], p.t.get("swa_scale"),
                                                 case.spec)
            pv = v4a.PagedViews(kv=kv, ix=ix, ring_main=ring_main, main_cap=main_cap, ring_ix=ring_ix,
                                ix_cap=ix_cap, ring_swa=ring_swa, swa_cap=swa_cap)
            self.layers.append(v4a.DeviceLayer(spec=p.spec, t=t, paged=pv,
                                               status=torch.zeros(1, dtype=torch.int32, device=device)))

    def _table(self, name: str, li: int):
        info = self.alloc.info(self.slot[name])
        off = info.table_offset + li * info.table_stride
        dev = self.tables[off: off + info.table_stride].view(-1, info.table_cols)
        return dev, self.alloc.table(self.slot[name], li), info

    def _paged_cache(self, name: str, li: int, dense_pool: torch.Tensor, dense_table: torch.Tensor) -> tuple:
        """Copies a dense case cache's blocks into the layer's pages; returns
        (pool, pages, device table, table columns)."""
        dev, host, info = self._table(name, li)
        bk = self.alloc.bucket(info.bucket)
        pool = self.pools[info.bucket]
        bt = dense_table.numpy()
        mask = bt >= 0
        src = torch.from_numpy(bt[mask].astype(np.int64)).to(pool.device)
        dst = torch.from_numpy(host[mask].astype(np.int64)).to(pool.device)
        pool.view(-1, bk.page_bytes)[dst] = dense_pool.view(-1, bk.page_bytes)[src]
        return pool, bk.num_pages, dev, info.table_cols

    def _paged_ring(self, name: str, li: int, rows: torch.Tensor, side, spec) -> tuple:
        """Copies a dense ring ([B][cap][row] plus an optional fp32 [B][cap])
        into the layer's ring pages: position p moves from slot p % cap to
        slot p % ring_cap.  Returns (v4a_ring_pages, ring_cap)."""
        dev, host, info = self._table(name, li)
        bk = self.alloc.bucket(info.bucket)
        pool = self.pools[info.bucket]
        Bn, cap = rows.shape[0], rows.shape[1]
        rb = rows[0, 0].numel() * rows.element_size()
        rows8 = rows.contiguous().view(torch.uint8).view(Bn, cap, rb)
        bi, sd, dr, ds = [], [], [], []
        for b in range(Bn):
            for pos in range(max(0, spec.cached[b] - cap), spec.cached[b]):
                sp = pos % info.ring_cap
                page, j = int(host[b, sp // info.slots]), sp % info.slots
                bi.append(b)
                sd.append(pos % cap)
                dr.append(page * bk.page_bytes + j * rb)
                ds.append(page * bk.page_bytes + info.slots * rb + 4 * j)
        if bi:
            d = pool.device
            bi_t, sd_t = torch.tensor(bi, device=d), torch.tensor(sd, device=d)
            off = torch.arange(rb, device=d)
            pool[torch.tensor(dr, device=d)[:, None] + off] = rows8[bi_t, sd_t]
            if side is not None and side.numel():
                side8 = side.contiguous().view(torch.uint8).view(Bn, cap, 4)
                pool[torch.tensor(ds, device=d)[:, None] + torch.arange(4, device=d)] = side8[bi_t, sd_t]
        rp = v4a.RingPages(pool.data_ptr(), bk.num_pages, bk.page_bytes, dev.data_ptr(), info.slots)
        return rp, info.ring_cap

    @property
    def tokens(self) -> int:
        """Query tokens per step (every layer sees the same batch)."""
        return self.layers[0].spec.tokens

    def run(self, stream=None):
        for st in self.steps:
            st.run(stream)

    def capture(self, stream) -> torch.cuda.CUDAGraph:
        """One CUDA graph of a whole step of the stack (run() once first, so
        that every layer's path is settled before capture)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run(torch.cuda.current_stream())
        return g

    def status(self) -> int:
        s = 0
        for L in self.layers:
            s |= int(L.status.item())
        return s

    def launches_per_step(self) -> int:
        return sum(st.launches_per_step() for st in self.steps)


def decode_1m_cases(seed: int = 0, c4a_case=None) -> dict:
    """The three layer kinds at 1M context, batch 4 (fp8 caches, fp4 indexer
    with per-32 fp32 scales, fp8 output); c4a_case may be given to reuse an
    already generated case of `c4a_decode_b4_1m`."""
    return {"c4a": c4a_case if c4a_case is not None else I.make_case(I.c4a_decode_1m(), seed),
            "c128a": I.make_case(I.c128a_decode_1m(), seed),
            "swa": I.make_case(I.swa_decode_1m(), seed)}


def shared_context_cases(seed: int = 0) -> dict:
    """Small cases of the three kinds with one context per sequence (the
    paged stack's rule), the queries normalised and rotated inside the step:
    sequence 0 at position 12,031 ends a c128a window and a c4a window,
    sequence 1 at 10,003 a c4a window only."""
    ctx = dict(batch=2, cached=(128 * 94 - 1, 4 * 2500 + 3), q_prep=True)
    c4a = dataclasses.replace(I.c4a_decode_1m(), name="paged_c4a_small", **ctx)
    c128a = dataclasses.replace(I.c128a_decode_1m(), name="paged_c128a_small", **ctx)
    swa = dataclasses.replace(I.swa_decode_1m(), name="paged_swa_small", **ctx)
    return {"c4a": I.make_case(c4a, seed), "c128a": I.make_case(c128a, seed), "swa": I.make_case(swa, seed)}


def shrink_cases(seed: int = 0) -> dict:
    """Small cases of the three kinds (a few thousand tokens of context), for tests."""
    c4a = dataclasses.replace(I.c4a_decode_1m(), name="stack_c4a_small", batch=2, cached=(4 * 3000 + 3, 9001))
    c128a = dataclasses.replace(I.c128a_decode_1m(), name="stack_c128a_small", batch=2, cached=(128 * 40 + 127, 7000))
    swa = dataclasses.replace(I.swa_decode_1m(), name="stack_swa_small", batch=2, cached=(5000, 77))
    return {"c4a": I.make_case(c4a, seed), "c128a": I.make_case(c128a, seed), "swa": I.make_case(swa, seed)}
