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


# --------------------------------------------------------------------------
# Window keys: rotated at their own positions
# --------------------------------------------------------------------------

def test_window_key_rotated_at_its_own_position_hand_values():
    """One key per position, a unit vector on a rope pair: the stored key is
    that pair rotated by exactly (position x the pair's frequency).  With
    rope_dims = 4 the pairs are (4, 5) at frequency 1 and (6, 7) at frequency
    10000^(-1/2) = 0.01.  cos/sin values from a table."""
    k = np.zeros((2, 8))
    k[0, 4] = k[1, 4] = 1.0
    out = L.window_keys(np.array([0, 0]), np.array([2, 3]), F.bf16_encode(k), 4, 10000.0)
    cos2, sin2 = -0.4161468365471424, 0.9092974268256817
    cos3, sin3 = -0.9899924966004454, 0.1411200080598672
    cos003, sin003 = 0.9995500337489875, 0.02999550020249566
    # two tokens of one call: each rotated at its own position, not the call's first or last
    assert np.allclose(out[(0, 2)], [0, 0, 0, 0, cos2, sin2, 0, 0], atol=1e-15)
    assert np.allclose(out[(0, 3)], [0, 0, 0, 0, cos3, sin3, 0, 0], atol=1e-15)
    k2 = np.zeros((2, 8))
    k2[0, 4] = 1.0
    k2[1, 6] = 1.0
    out2 = L.window_keys(np.array([0, 1]), np.array([3, 3]), F.bf16_encode(k2), 4, 10000.0)
    assert np.allclose(out2[(0, 3)], [0, 0, 0, 0, cos3, sin3, 0, 0], atol=1e-15)
    assert np.allclose(out2[(1, 3)], [0, 0, 0, 0, 0, 0, cos003, sin003], atol=1e-15)


def _window_chain(delta: int):
    """The oracle's chain for the last query of one call of 160 tokens at
    positions 256 + delta ..: the call's compressed entries (compress) and
    window keys (window_keys) as keys, fp64 attention, inverse RoPE.  Every
    random draw is independent of delta."""
    from oracle import attention as A
    from oracle import compressor as Cm
    rng = np.random.default_rng(21)
    D, R, th, H, n_new, P0 = 64, 32, 10000.0, 2, 160, 256
    cap = 8 - 1 + n_new
    x = F.bf16_encode(rng.standard_normal((n_new, D)))
    g = rng.standard_normal(n_new)
    bias, gamma = rng.normal(0, 0.5, 8), 1 + rng.normal(0, 0.1, D)
    older, older_g = F.bf16_encode(rng.standard_normal((4, D))), rng.standard_normal(4)
    kw = F.bf16_encode(rng.standard_normal((n_new, D)))
    qt = rng.standard_normal((H, D))
    ring_x, ring_g = np.zeros((1, cap, D), np.uint16), np.zeros((1, cap))
    for j in range(4):                                   # positions 252 + delta .. 255 + delta
        p = P0 + delta - 4 + j
        ring_x[0, p % cap], ring_g[0, p % cap] = older[j], older_g[j]
    comp = L.Compressor(4, D, R, th, bias, gamma, ring_x, ring_g)
    pos = np.arange(P0 + delta, P0 + delta + n_new)
    seq = np.zeros(n_new, int)
    entries = L.compress(seq, pos, x, g, comp)
    win = L.window_keys(seq, pos, kw, R, th)
    m = int(pos[-1])
    keys = [v for (_, i), v in sorted(entries.items()) if G.anchor(i, 4) <= m]
    keys += [win[(0, p)] for p in G.swa_positions(m, 128)]
    assert len(keys) == n_new // 4 + 128
    o, _ = A.shared_kv_attention(Cm.rope(qt, m, R, th), np.stack(keys), 1 / math.sqrt(D))
    return A.inverse_rope(o, m, R, th)


def test_window_keys_translation_invariance_through_the_layer_chain(monkeypatch):
    """Shifting every position of the call (query, compressed anchors, window
    keys) by a multiple of 256 leaves R_m^{-1} o_m unchanged to fp64 round-off
    ("DeepSeek V4 in vLLM", appendix "why inverse RoPE": the output depends on
    relative positions only).  Negative control: window keys left unrotated."""
    base = _window_chain(0)
    for delta in (256, 768, 1 << 20):
        assert np.allclose(_window_chain(delta), base, atol=1e-10)
    monkeypatch.setattr(L, "rope", lambda v, pos, rope_dims, theta, inverse=False: v)
    assert not np.allclose(_window_chain(768), _window_chain(0), atol=1e-3)


# --------------------------------------------------------------------------
# The queries' elementwise work (fusion (3): Q norm, then the query rotated
# at its position like every key)
# --------------------------------------------------------------------------

def test_query_prep_hand_worked_example():
    """D = 4, one head at position 0 (no rotation), eps 0: q = (1, 2, 2, 4) has
    mean square 25/4, so the normalised row is (0.4, 0.8, 0.8, 1.6); times
    gamma (1, 0.5, 2, 1) it is (0.4, 0.4, 1.6, 1.6)."""
    from oracle import layer as LY
    q = F.bf16_encode(np.array([[[1.0, 2.0, 2.0, 4.0]]]))
    out = LY.query_prep(q, np.array([0]), np.array([1.0, 0.5, 2.0, 1.0]), 2, 10000.0, eps=0.0)
    assert np.allclose(out[0, 0], [0.4, 0.4, 1.6, 1.6], rtol=0, atol=1e-15)


def test_query_prep_normalises_each_head_on_its_own():
    """gamma = 1, eps = 0: every (token, head) row has RMS 1 after the norm and
    the rotation (which keeps lengths), whatever the heads' magnitudes."""
    from oracle import layer as LY
    rng = np.random.default_rng(3)
    D, H = 64, 5
    q = rng.standard_normal((2, H, D)) * np.array([1e-3, 1.0, 30.0, 7.0, 0.2])[None, :, None]
    out = LY.query_prep(F.bf16_encode(q), np.array([17, 900]), np.ones(D), 32, 10000.0, eps=0.0)
    rms = np.sqrt(np.mean(out ** 2, axis=-1))
    assert np.allclose(rms, 1.0, rtol=1e-12)


def test_query_prep_scores_depend_on_relative_position_only():
    """With a gamma that differs inside each rotary pair, q . k of a prepared
    query at m and a key rotated at n is unchanged when m and n move
    together, and changes when only m moves (a query left unrotated, rotated
    the wrong way or rotated before the norm fails this)."""
    from oracle import layer as LY
    from oracle import compressor as CO
    rng = np.random.default_rng(5)
    D, R = 128, 64
    gamma = 1.0 + 0.3 * rng.standard_normal(D)
    q = F.bf16_encode(rng.standard_normal((1, 1, D)))
    k = rng.standard_normal(D)

    def score(m, n):
        return float(LY.query_prep(q, np.array([m]), gamma, R, 10000.0)[0, 0] @ CO.rope(k, n, R, 10000.0))

    base = score(1000, 37)
    assert abs(score(1000 + 4321, 37 + 4321) - base) < 1e-9 * (1 + abs(base))
    assert abs(score(1000 + 4321, 37) - base) > 1e-3


# --------------------------------------------------------------------------
# The indexer query's preparation (RoPE, per-head fp8, weight multiply)
# --------------------------------------------------------------------------

def test_index_query_prep_hand_worked_example():
    """Position 0 (no rotation): q = (1, 2, 2, 4) has amax 4, so the scale is
    4/448 and the codes are e4m3 of (112, 224, 224, 448), all exact; the
    weights are multiplied by w_mult."""
    from oracle import layer as LY
    q = F.bf16_encode(np.array([[[1.0, 2.0, 2.0, 4.0]]]))
    codes, sc, w = LY.index_query_prep(q, np.array([0]), np.array([[0.75]]), 0.125, 2, 10000.0)
    assert sc[0, 0] == np.float32(4.0 / 448.0)
    assert list(F.e4m3_decode(codes[0, 0])) == [112.0, 224.0, 224.0, 448.0]
    assert w[0, 0] == 0.75 * 0.125


def test_index_query_prep_rotates_forward_per_head():
    """Decoding the codes and rotating back by the token's position gives the
    bf16 query within one e4m3 step of the row (the two errors of a pair
    mix); a rotation the wrong way, at the wrong position or on the wrong
    dims fails.  Each head has its own scale, amax / 448 of its rotated row."""
    from oracle import layer as LY
    from oracle import compressor as CO
    rng = np.random.default_rng(9)
    T, H, D, R = 3, 4, 128, 64
    q = rng.standard_normal((T, H, D)) * np.array([0.01, 1.0, 5.0, 80.0])[None, :, None]
    qb = F.bf16_encode(q)
    pos = np.array([5, 1000, 777_777])
    codes, sc, _ = LY.index_query_prep(qb, pos, np.ones((T, H)), 1.0, R, 10000.0)
    qd = F.bf16_decode(qb)
    for t in range(T):
        for h in range(H):
            rot = CO.rope(qd[t, h], int(pos[t]), R, 10000.0)
            assert sc[t, h] == np.float32(np.max(np.abs(rot)) / 448.0)
            back = CO.rope(F.e4m3_decode(codes[t, h]) * sc[t, h], int(pos[t]), R, 10000.0, inverse=True)
            step = F.e4m3_ulp(rot / sc[t, h]) * sc[t, h]
            assert np.all(np.abs(back - qd[t, h]) <= np.max(step) + 1e-12)
    assert len(set(np.round(sc[0], 12))) == H
