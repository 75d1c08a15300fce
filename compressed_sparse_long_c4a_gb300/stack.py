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

Each layer owns its caches, rings and workspaces (built from one synthetic
case per layer kind and copied per layer), so a replay of the graph is one
decode step of the whole attention stack: every layer inserts its new
entries and attends over its own caches.
"""
from __future__ import annotations

import dataclasses

import torch

from . import inputs as I
from . import v4a


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

    def __init__(self, kinds: list, cases: dict, device="cuda", overlap: str = "serial"):
        self.kinds = list(kinds)
        self.layers = []
        self.steps = []
        proto = {}
        for k in set(self.kinds):
            proto[k] = v4a.DeviceLayer.from_case(cases[k], device)
        for k in self.kinds:
            p = proto[k]
            L = v4a.DeviceLayer(spec=p.spec, t={n: x.clone() for n, x in p.t.items()},
                                status=torch.zeros(1, dtype=torch.int32, device=p.status.device))
            self.layers.append(L)
            self.steps.append(v4a.Step(L, overlap=overlap if k == "c4a" else "serial"))
        del proto

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


def shrink_cases(seed: int = 0) -> dict:
    """Small cases of the three kinds (a few thousand tokens of context), for tests."""
    c4a = dataclasses.replace(I.c4a_decode_1m(), name="stack_c4a_small", batch=2, cached=(4 * 3000 + 3, 9001))
    c128a = dataclasses.replace(I.c128a_decode_1m(), name="stack_c128a_small", batch=2, cached=(128 * 40 + 127, 7000))
    swa = dataclasses.replace(I.swa_decode_1m(), name="stack_swa_small", batch=2, cached=(5000, 77))
    return {"c4a": I.make_case(c4a, seed), "c128a": I.make_case(c128a, seed), "swa": I.make_case(swa, seed)}
