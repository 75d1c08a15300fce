"""Feeds a seeded workload (``inputs.Case``) to the fp64 oracle.

Test-side glue only: converts torch CPU tensors to the numpy bit patterns the
oracle reads, and runs the oracle's stages in step order.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import formats as F
from oracle import geometry as G
from oracle import layer as L


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.double().numpy()


def main_compressor(case) -> L.Compressor:
    s = case.spec
    return L.Compressor(ratio=s.ratio, dim=s.dim, rope_dims=s.rope_dims, theta=s.theta,
                        bias=f64(case.bias), gamma=f64(case.gamma),
                        ring_x=u16(case.ring_x), ring_gate=f64(case.ring_gate))


def indexer_compressor(case) -> L.Compressor:
    s = case.spec
    return L.Compressor(ratio=4, dim=s.ix_dim, rope_dims=s.ix_rope_dims, theta=s.theta,
                        bias=f64(case.bias_i), gamma=f64(case.gamma_i),
                        ring_x=u16(case.ring_x_i), ring_gate=f64(case.ring_gate_i))


def oracle_compress(case):
    """-> (main entries {(b,i): vec}, indexer entries, window keys {(b,p): vec})."""
    s = case.spec
    sid, pos = case.seq_ids.numpy(), case.positions.numpy()
    main = L.compress(sid, pos, u16(case.x), f64(case.gate), main_compressor(case))
    ix = {}
    if s.ix_heads:
        ix = L.compress(sid, pos, u16(case.x_i), f64(case.gate_i), indexer_compressor(case))
    swa = L.window_keys(sid, pos, u16(case.k_swa), s.rope_dims, s.theta)
    return main, ix, swa


def oracle_state_after_compress(case, main, ix, swa):
    """The oracle's own copy of pools and window ring after inserting."""
    s = case.spec
    kv = u8(case.kv_pool).copy()
    bt = case.block_table.numpy()
    for (b, i), v in main.items():
        blk, slot = G.slot_of(bt[b], i, s.ratio)
        L.write_kv_entry(kv, s.kv_block_bytes, blk, slot, v, s.kv_fmt, s.entries_per_block, s.dim)
    ixp = None
    if s.ix_heads:
        ixp = u8(case.ix_pool).copy()
        for (b, i), v in ix.items():
            blk, slot = G.slot_of(bt[b], i, 4)
            L.write_ix_entry(ixp, s.ix_block_bytes, blk, slot, v, s.ix_fmt, s.ix_dim)
    if s.swa_fmt == F.KV_BF16:
        ring = u16(case.swa_ring).copy()
        rsc = None
    else:
        ring = u8(case.swa_ring).copy()
        rsc = case.swa_scale.double().numpy().copy()
    cap = ring.shape[1]
    for (b, p), v in swa.items():
        data, sc = L.encode_kv_row(v, s.swa_fmt)
        if s.swa_fmt == F.KV_BF16:
            ring[b, p % cap] = data.view(np.uint16)
        else:
            ring[b, p % cap] = data
            rsc[b, p % cap] = sc
    return kv, ixp, ring, rsc


def step_index_query(case):
    """The indexer query, its scales and head weights a whole step's scan
    reads: the oracle's own preparation (RoPE + per-head fp8 + weights) when
    the step prepares them, else the case's inputs."""
    s = case.spec
    if s.ix_q_prep:
        return L.index_query_prep(u16(case.q_i_raw), case.positions.numpy(), f64(case.w_i_raw), s.ix_w_mult,
                                  s.ix_rope_dims, s.theta)
    return (u16(case.q_i) if s.ix_q_fmt == 0 else u8(case.q_i)), f64(case.q_i_scale), f64(case.w_i)


def oracle_index(case, ix_pool, rows=None, query=None):
    """Indexer scores and top-k of the case's queries (query: a (q, q_scale,
    weights) triple to use instead of the case's inputs)."""
    s = case.spec
    if query is None:
        query = ((u16(case.q_i) if s.ix_q_fmt == 0 else u8(case.q_i)), f64(case.q_i_scale), f64(case.w_i))
    q, qs, w = query
    return L.index_topk(case.seq_ids.numpy(), case.positions.numpy(), q, qs, w, s.ix_q_fmt == 1,
                        ix_pool, s.ix_block_bytes, case.block_table.numpy(), s.ix_fmt,
                        s.ix_dim, s.topk, rows=rows)


def oracle_query(case):
    """The oracle's prepared queries (norm + RoPE, fusion (3)) in float64."""
    s = case.spec
    return L.query_prep(u16(case.q_raw), case.positions.numpy(), f64(case.gamma_q), s.rope_dims, s.theta)


def step_q_bits(case):
    """The bf16 query a whole step's attention reads: the oracle's prepared
    query rounded to bf16 when the step prepares it, else the case's q."""
    if case.spec.q_prep:
        return F.bf16_encode(oracle_query(case))
    return u16(case.q)


def oracle_attention(case, kv_pool, swa_ring, swa_scale, idx, rows=None, q_bits=None):
    """Attention of the case's queries (q_bits: the bf16 query to use instead
    of case.q, e.g. the step's prepared query)."""
    s = case.spec
    q = u16(case.q) if q_bits is None else q_bits
    return L.attention(case.seq_ids.numpy(), case.positions.numpy(), q, idx,
                       kv_pool, s.kv_block_bytes, case.block_table.numpy(), s.kv_fmt, s.ratio,
                       s.dim, swa_ring, swa_scale, s.swa_fmt, s.swa, 1.0 / math.sqrt(s.dim),
                       rows=rows)


def oracle_output(case, o_bits):
    s = case.spec
    return L.output_stage(o_bits, case.positions.numpy(), s.rope_dims, s.theta, s.out_fmt == 1)
