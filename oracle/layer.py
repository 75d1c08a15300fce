"""One layer step of compressed sparse attention, composed from the stages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Order of the stages within a step ("DeepSeek V4 in vLLM", Method details,
"keeping the GPU busy"): compress + RMSNorm + RoPE + cache insert (main and
indexer), RoPE + insert of the window key; indexer scoring and top-k; sparse
attention over the selected entries plus the window; inverse RoPE (+ fp8).

Conventions taken where the page is silent:
* Rings: the compressor keeps the raw (x_t, g_t) of its last positions in a
  per-sequence ring indexed by position mod capacity; the window ring keeps
  the rotated (and encoded) key of each position at position mod capacity.
  New tokens of one call are read from the call's inputs, older positions
  from the rings.
* Causality inside a chunk: a query at m sees every entry with anchor <= m,
  including entries emitted earlier in the same call, and window tokens
  written in the same call.

All arrays are numpy; bf16 tensors are passed as uint16 bit patterns and fp8 /
fp4 data as uint8 bytes, exactly as they sit in device memory.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import formats as F
from . import geometry as G
from .compressor import compressed_entry, rms_norm, rope, RMS_EPS
from .indexer import index_scores, topk_set
from .attention import shared_kv_attention, inverse_rope, quant_fp8_per_token


@dataclass
class Compressor:
    """Per-layer compressor parameters and its ring (one for main, one for indexer)."""
    ratio: int
    dim: int
    rope_dims: int
    theta: float
    bias: np.ndarray       # [window] fp64
    gamma: np.ndarray      # [dim] fp64
    ring_x: np.ndarray     # [B][cap][dim] uint16 (bf16 bits)
    ring_gate: np.ndarray  # [B][cap] float


def _token_rows(seq_ids, positions):
    return {(int(b), int(p)): t for t, (b, p) in enumerate(zip(seq_ids, positions))}


def compress(seq_ids, positions, x_bits, gate, comp: Compressor) -> dict:
    """Entries emitted by this call: {(seq, entry index): float64 vector}."""
    rows = _token_rows(seq_ids, positions)
    cap = comp.ring_x.shape[1]

    def x_of(b, p):
        t = rows.get((b, p))
        if t is not None:
            return F.bf16_decode(x_bits[t])
        return F.bf16_decode(comp.ring_x[b, p % cap])

    def g_of(b, p):
        t = rows.get((b, p))
        if t is not None:
            return float(gate[t])
        return float(comp.ring_gate[b, p % cap])

    out = {}
    for b, p in zip(seq_ids, positions):
        b, p = int(b), int(p)
        i = G.emits_at(p, comp.ratio)
        if i is None:
            continue
        out[(b, i)] = compressed_entry(lambda q: x_of(b, q), lambda q: g_of(b, q), i,
                                       comp.ratio, comp.bias, comp.gamma,
                                       comp.rope_dims, comp.theta)
    return out


def window_keys(seq_ids, positions, k_bits, rope_dims, theta) -> dict:
    """Rotated window keys of this call's tokens: {(seq, position): vector}."""
    return {(int(b), int(p)): rope(F.bf16_decode(k_bits[t]), int(p), rope_dims, theta)
            for t, (b, p) in enumerate(zip(seq_ids, positions))}

def query_prep(q_bits, positions, gamma, rope_dims, theta, eps=RMS_EPS) -> np.ndarray:
    """The queries' elementwise work before attention ("DeepSeek V4 in vLLM",
    Method details, fusion (3): the Q norm, horizontally fused with the window
    keys' RoPE + insert).  Reading: each (token, head) row of the bf16 query
    is RMS-normalised over the head's dims with the shared weight gamma, then
    rotated at the token's position like every key (last rope_dims dims,
    interleaved pairs), so that q . k depends on the relative position only.
    q_bits: [T][H][D] bf16 bits -> float64 [T][H][D]."""
    q = F.bf16_decode(q_bits)
    out = np.empty_like(q)
    for t in range(q.shape[0]):
        for h in range(q.shape[1]):
            out[t, h] = rope(rms_norm(q[t, h], gamma, eps), int(positions[t]), rope_dims, theta)
    return out

def index_query_prep(q_bits, positions, w, w_mult, rope_dims, theta):
    """The indexer query's preparation ("DeepSeek V4 in vLLM", Method details:
    the reused DeepSeek-V3.2 fusion of Q RoPE, quantisation and the weight
    multiplication).  Reading: each (token, head) row of the bf16 indexer
    query is rotated at the token's position on its last rope_dims dims, then
    encoded as e4m3 with one scale per (token, head), amax / 448 (the scan's
    fp8 query format); the head weights are multiplied by the constant
    w_mult.  -> (codes uint8 [T][H][D], scales float64 [T][H], weights
    float64 [T][H])."""
    q = F.bf16_decode(q_bits)
    T, H, D = q.shape
    codes = np.empty((T, H, D), np.uint8)
    scales = np.empty((T, H), np.float64)
    for t in range(T):
        for h in range(H):
            codes[t, h], scales[t, h] = F.fp8_token_encode(rope(q[t, h], int(positions[t]), rope_dims, theta))
    return codes, scales, np.asarray(w, np.float64) * float(w_mult)

# --------------------------------------------------------------------------
# Encoding into the oracle's own copy of the caches
# --------------------------------------------------------------------------

def encode_kv_row(v: np.ndarray, fmt: int):
    """-> (data bytes, scale or None) of one shared-KV / window row (the
    DeepSeek-V4 row carries its scales inside its 584 bytes)."""
    if fmt == F.KV_BF16:
        return F.bf16_encode(v).view(np.uint8), None
    if fmt == F.KV_FP8_DSV4:
        return F.dsv4_row_encode(v), None
    codes, s = F.fp8_token_encode(v)
    return codes, s


def encode_ix_row(v: np.ndarray, fmt: int):
    if fmt == F.IX_BF16:
        return F.bf16_encode(v).view(np.uint8), None
    if fmt == F.IX_FP8_B128:
        return F.fp8_blocks_encode(v, 128)
    if fmt == F.IX_FP4_MX32:
        return F.fp4_mx_blocks_encode(v, 32)
    return F.fp4_blocks_encode(v, 32)


def write_kv_entry(pool: np.ndarray, block_bytes: int, blk: int, slot: int, v, fmt,
                   entries: int, dim: int):
    data, s = encode_kv_row(v, fmt)
    base = blk * block_bytes
    row = data.shape[0]
    pool[base + slot * row: base + (slot + 1) * row] = data
    if s is not None:
        off = base + entries * dim + 4 * slot
        pool[off:off + 4] = np.array([s], np.float32).view(np.uint8)


def write_ix_entry(pool: np.ndarray, block_bytes: int, blk: int, slot: int, v, fmt, dim: int):
    data, sc = encode_ix_row(v, fmt)
    base = blk * block_bytes
    row = data.shape[0]
    pool[base + slot * row: base + (slot + 1) * row] = data
    if sc is not None:
        sc = np.asarray(sc, np.float32).reshape(-1)
        off = base + 64 * row + 4 * sc.shape[0] * slot
        pool[off:off + 4 * sc.shape[0]] = sc.view(np.uint8)

# --------------------------------------------------------------------------
# Reading visible entries
# --------------------------------------------------------------------------

def visible_kv(pool, block_bytes, bt_row, n, fmt, ratio, dim) -> np.ndarray:
    """Decoded entries 0..n-1 of one sequence's shared-KV cache -> [n][dim]."""
    e = G.entries_per_block(ratio)
    nblk = (n + e - 1) // e
    if nblk == 0:
        return np.zeros((0, dim))
    blocks = np.asarray(bt_row[:nblk], np.int64)
    raw = pool.reshape(-1, block_bytes)[blocks]
    return F.kv_block_decode(raw, fmt, e, dim).reshape(nblk * e, dim)[:n]


def visible_ix(pool, block_bytes, bt_row, n, fmt, dim) -> np.ndarray:
    nblk = (n + 63) // 64
    if nblk == 0:
        return np.zeros((0, dim))
    blocks = np.asarray(bt_row[:nblk], np.int64)
    raw = pool.reshape(-1, block_bytes)[blocks]
    return F.ix_block_decode(raw, fmt, dim).reshape(nblk * 64, dim)[:n]


def swa_row(ring, ring_scale, b, p, fmt) -> np.ndarray:
    cap = ring.shape[1]
    if fmt == F.KV_BF16:
        return F.bf16_decode(ring[b, p % cap])
    return F.e4m3_decode(ring[b, p % cap]) * float(ring_scale[b, p % cap])

# --------------------------------------------------------------------------
# Stages over a batch
# --------------------------------------------------------------------------

def index_topk(seq_ids, positions, q_i, q_i_scale, w, q_fp8: bool, ix_pool, ix_block_bytes,
               block_table, ix_fmt, ix_dim, k, rows=None):
    """-> (idx [T][k] int64 ascending with -1 padding, scores list per query)."""
    T = len(positions)
    rows = range(T) if rows is None else rows
    keys_cache = {}
    idx = {}
    scores = {}
    for t in rows:
        b, m = int(seq_ids[t]), int(positions[t])
        n = G.n_visible(m, 4)
        if b not in keys_cache or keys_cache[b].shape[0] < n:
            nmax = max(G.n_visible(int(pp), 4) for bb, pp in zip(seq_ids, positions) if int(bb) == b)
            keys_cache[b] = visible_ix(ix_pool, ix_block_bytes, block_table[b], nmax, ix_fmt, ix_dim)
        keys = keys_cache[b][:n]
        if q_fp8:
            q = F.e4m3_decode(q_i[t]) * np.asarray(q_i_scale[t], np.float64)[:, None]
        else:
            q = F.bf16_decode(q_i[t])
        s = index_scores(q, np.asarray(w[t], np.float64), keys)
        scores[t] = s
        idx[t] = topk_set(s, k)
    return idx, scores


def attention(seq_ids, positions, q_bits, idx, kv_pool, kv_block_bytes, block_table, kv_fmt,
              ratio, dim, swa_ring, swa_scale, swa_fmt, window, tau, rows=None):
    """-> {t: (o [H][D] float64, lse [H])}.  idx[t] None means 'all visible'."""
    T = len(positions)
    rows = range(T) if rows is None else rows
    out = {}
    for t in rows:
        b, m = int(seq_ids[t]), int(positions[t])
        n = G.n_visible(m, ratio)
        ent = visible_kv(kv_pool, kv_block_bytes, block_table[b], n, kv_fmt, ratio, dim)
        sel = np.arange(n) if idx is None or idx[t] is None else \
            np.asarray([i for i in idx[t] if i >= 0], np.int64)
        keys_c = ent[sel]
        keys_w = np.stack([swa_row(swa_ring, swa_scale, b, p, swa_fmt)
                           for p in G.swa_positions(m, window)])
        keys = np.concatenate([keys_c, keys_w], axis=0)
        q = F.bf16_decode(q_bits[t])
        out[t] = shared_kv_attention(q, keys, tau)
    return out


def output_stage(o_bits, positions, rope_dims, theta, fp8: bool):
    """-> list of (rotated o [H][D] float64, codes or None, scale or None)."""
    res = []
    for t, m in enumerate(positions):
        o = inverse_rope(F.bf16_decode(o_bits[t]), int(m), rope_dims, theta)
        if fp8:
            codes, s = quant_fp8_per_token(o)
            res.append((o, codes, s))
        else:
            res.append((o, None, None))
    return res
