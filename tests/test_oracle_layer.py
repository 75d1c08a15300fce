"""Pins of the oracle's batch-level stages: paged gather by brute force, the
dense special case of the full attention stage against torch fp64, window
coverage, and the workload generator's structure."""
import math

import numpy as np
import torch

from compressed_sparse_long_c4a_gb300 import inputs as I
from oracle import formats as F
from oracle import geometry as G
from oracle import layer as L
from tests import oracle_bridge as OB


def _tiny(ratio=4, **kw):
    base = dict(name="tiny", ratio=ratio, batch=3, heads=4, dim=128, cached=(300, 517, 1030),
                ix_heads=4, ix_dim=64, ix_fmt=I.IX_BF16, topk=16)
    if ratio == 128:
        base.update(ix_heads=0, ix_dim=0, topk=0)
    base.update(kw)
    return I.LayerSpec(**base)


def test_visible_kv_gathers_by_block_table():
    case = I.make_case(_tiny(), seed=3)
    s = case.spec
    pool = OB.u8(case.kv_pool)
    bt = case.block_table.numpy()
    for b in range(s.batch):
        n = G.n_visible(s.cached[b], 4)
        got = L.visible_kv(pool, s.kv_block_bytes, bt[b], n, s.kv_fmt, 4, s.dim)
        for i in range(0, n, 7):
            blk, slot = G.slot_of(bt[b], i, 4)
            off = blk * s.kv_block_bytes + slot * s.dim * 2
            ref = F.bf16_decode(pool[off:off + s.dim * 2].copy().view(np.uint16))
            assert np.array_equal(got[i], ref)


def test_attention_stage_dense_case_against_torch():
    case = I.make_case(_tiny(ratio=128, cached=(100, 300, 700)), seed=4)
    s = case.spec
    kv, _, ring, rsc = OB.oracle_state_after_compress(case, *OB.oracle_compress(case))
    out = OB.oracle_attention(case, kv, ring, rsc, idx=None)
    bt = case.block_table.numpy()
    for t in range(s.tokens):
        b, m = int(case.seq_ids[t]), int(case.positions[t])
        n = G.n_visible(m, 128)
        rows = []
        for i in range(n):
            blk, slot = G.slot_of(bt[b], i, 128)
            off = blk * s.kv_block_bytes + slot * s.dim * 2
            rows.append(F.bf16_decode(kv[off:off + 2 * s.dim].copy().view(np.uint16)))
        cap = ring.shape[1]
        for p in range(max(0, m - 127), m + 1):
            rows.append(F.bf16_decode(ring[b, p % cap]))
        keys = torch.from_numpy(np.stack(rows))
        q = torch.from_numpy(F.bf16_decode(OB.u16(case.q[t])))
        ref = torch.softmax(q @ keys.T / math.sqrt(s.dim), dim=-1) @ keys
        assert np.allclose(out[t][0], ref.numpy(), atol=1e-12)
        if m < 127:
            assert n == 0 and len(rows) == m + 1


def test_index_stage_matches_brute_force_scores():
    case = I.make_case(_tiny(), seed=5)
    s = case.spec
    _, ixe, _ = OB.oracle_compress(case)
    _, ixp, _, _ = OB.oracle_state_after_compress(case, *OB.oracle_compress(case))
    idx, scores = OB.oracle_index(case, ixp)
    bt = case.block_table.numpy()
    for t in range(s.tokens):
        b, m = int(case.seq_ids[t]), int(case.positions[t])
        n = G.n_visible(m, 4)
        assert scores[t].shape == (n,)
        q = F.bf16_decode(OB.u16(case.q_i[t]))
        w = case.w_i[t].double().numpy()
        for i in (0, n // 2, n - 1):
            blk, slot = G.slot_of(bt[b], i, 4)
            off = blk * s.ix_block_bytes + slot * s.ix_dim * 2
            k = F.bf16_decode(ixp[off:off + 2 * s.ix_dim].copy().view(np.uint16))
            ref = sum(w[h] * max(0.0, float(q[h] @ k)) for h in range(s.ix_heads))
            assert math.isclose(scores[t][i], ref, rel_tol=1e-12, abs_tol=1e-12)
        sel = idx[t]
        assert len(set(sel.tolist())) == s.topk and sel.max() < n


def test_generator_structure():
    for name, fn in I.WORKLOADS.items():
        spec = fn()
        assert spec.entries_per_block * spec.ratio == 256
        if spec.ratio == 4 and spec.new == 1:
            assert spec.ring_cap == 8
    s = I.c4a_decode_1m()
    assert s.cached[0] == (1 << 20) - 1 and G.emits_at(s.cached[0], 4) == 262143
    assert G.n_visible(s.cached[0], 4) == 262144 == s.max_blocks * 64
    s2 = I.c4a_decode_b32_32k_64k()
    m = s2.cached
    assert G.emits_at(m[0], 4) is not None
    assert G.emits_at(m[1], 4) % 64 == 0 and G.emits_at(m[2], 4) % 64 == 63 and m[3] % 256 == 0
    assert all(32768 <= v <= 65536 for v in m)
    case = I.make_case(_tiny(), seed=0)
    bt = case.block_table
    used = bt[bt >= 0]
    assert used.unique().numel() == used.numel()
